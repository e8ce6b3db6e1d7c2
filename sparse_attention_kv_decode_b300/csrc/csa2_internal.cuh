// Internal declarations and device helpers of libcsa2 (sm_103a only).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the caller's workspace pointer)
//   [0, 256)   header: device status word (u32) at offset 0
//   [256, ..)  scratch of csa2_index_topk: fp32 indexer scores [Q][n_pad]
//              (calls on one workspace are stream-ordered). The attention calls
//              use only the status word: their splits merge on chip.
// ---------------------------------------------------------------------------
constexpr size_t kWsHeader = 256;
constexpr int kMaxSplits = 16;  // power-of-two key splits per query (one cluster)
constexpr int kScoreTile = 1024;  // keys per indexer CTA
constexpr int kMaxK = 4096;
constexpr int64_t kMaxNStride = 262144;  // 1M tokens at 4:1
constexpr int kMaxWin = 256;

inline int64_t score_pad(int64_t n) { return (n + kScoreTile - 1) / kScoreTile * kScoreTile; }

// Number of key splits per query for the sparse attention (about one wave of
// CTAs when the batch is small; one split per query when there are many).
int attn_splits(int64_t Q, int K, int W, int n_sm);


// Per-query score range words (two uint32 per query) that the scoring kernel
// leaves for the selection; they sit right after the header, at a fixed offset
// per query, and the selection sets them back to zero.
inline size_t range_bytes(int64_t Q) { return ((size_t)Q * 8 + 255) / 256 * 256; }
// candidate pool of a REINDEX call: block ids [Q][K] and the visible count per query
inline size_t pool_bytes(int64_t Q, int K) {
  return ((size_t)Q * K * 4 + 255) / 256 * 256 + ((size_t)Q * 4 + 255) / 256 * 256;
}
inline size_t scores_bytes(int64_t Q, int64_t n_stride) {
  return (size_t)Q * (size_t)score_pad(n_stride) * 4;
}

int device_sm_count();

// Sets a kernel attribute once per (device, slot): launchers call this instead of
// cudaFuncSetAttribute so that no attribute call happens while a stream is
// being captured into a CUDA graph (after the first, eager, call on a device).
cudaError_t set_attr_once(int slot, const void* fn, cudaFuncAttribute attr, int value);

// 2-D bf16 tensor map (row-major [outer][inner], 128-byte swizzle, zero fill
// outside the tensor) for TMA tile loads of box_outer rows x box_inner columns.
bool encode_tensor_map_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                               uint32_t box_inner, uint32_t box_outer);

// Kernel launchers (return cudaError_t of the launch).
cudaError_t launch_wait_check(uint64_t limit_ns, uint32_t* status, cudaStream_t st);
cudaError_t launch_cache_append(int B, int32_t* n_tokens, int advance, int ratio, const void* swa_row,
                                void* swa_kv, int64_t s_stride, int n_win, const void* entry_kv,
                                int entry_dtype, const void* entry_z, uint8_t* codes, uint8_t* scales,
                                void* z, int64_t n_stride, int32_t* n_visible, int32_t* win_start,
                                int32_t* win_len, uint32_t* status, cudaStream_t st);
cudaError_t launch_encode_quant(const void* h, int h_dtype, int64_t rows, uint8_t* codes,
                                uint8_t* scales, cudaStream_t st);
// pool / pool_nv / pool_stride (nullable): score the positions of a candidate pool
// (ascending block ids [Q][pool_stride], visible positions per query) instead of 0..n-1
cudaError_t launch_index_score(const void* q_idx, const float* w_idx, const void* z,
                               int64_t n_stride, const int32_t* n_visible, int B, int T, int H_I,
                               float* scores, int64_t score_stride, uint32_t* range,
                               uint32_t* status, cudaStream_t st, const int32_t* pool = nullptr,
                               const int32_t* pool_nv = nullptr, int pool_stride = 0);
// Indexer scoring of T >= 256 / H_I query tokens per sequence as a tcgen05 GEMM (keys x
// (token, head) tiles); same scores and range words as launch_index_score without a pool.
bool index_gemm_applies(int T, int H_I);
bool index_stream_applies(int B, int T, int H_I);
cudaError_t launch_index_stream(const void* q_idx, const float* w_idx, const void* z, int64_t n_stride,
                                const int32_t* n_visible, int B, int T, int H_I, float* scores,
                                int64_t score_stride, uint32_t* range, uint32_t* status, cudaStream_t st);
cudaError_t launch_index_gemm(const void* q_idx, const float* w_idx, const void* z, int64_t n_stride,
                              const int32_t* n_visible, int B, int T, int H_I, float* scores,
                              int64_t score_stride, uint32_t* range, uint32_t* status, cudaStream_t st);
// pf_codes / pf_scales (nullable): FP4 cache whose rows of the selected entries are
// requested into L2 as they are written (batch b = query / T, rows of n_stride)
cudaError_t launch_topk_select(const float* scores, int64_t score_stride, const int32_t* n_visible,
                               int Q, int64_t n_stride, int K, uint32_t* range, int32_t* out_idx,
                               float* out_scores, uint32_t* status, cudaStream_t st,
                               const uint8_t* pf_codes = nullptr, const uint8_t* pf_scales = nullptr,
                               int T = 1, int64_t kv_stride = -1, const int32_t* pool = nullptr,
                               int pool_stride = 0);
// Candidate pool of the Hierarchical Sparse Indexer from a selection sel [Q][K]:
// ascending block ids blocks [Q][K] and the number of pool positions below n_visible
cudaError_t launch_pool_build(const int32_t* sel, int Q, int K, const int32_t* n_visible, int64_t n_stride,
                              int32_t* blocks, int32_t* pool_nv, uint32_t* status, cudaStream_t st);
cudaError_t launch_copy_idx(const int32_t* src, int32_t* dst, int64_t n, cudaStream_t st);
cudaError_t launch_sparse_attn(int B, int T, int H, const void* q, const uint8_t* codes,
                               const uint8_t* scales, int64_t n_stride, const int32_t* idx,
                               int K, float scale_log2, float* o_g, float* lse_g, int nsplit,
                               float* xchg, uint32_t* status, cudaStream_t st);
cudaError_t launch_swa_merge(int B, int T, int H, const void* q, const void* swa,
                             int64_t s_stride, const int32_t* win_start, const int32_t* win_len,
                             int n_win, float scale_log2, const float* o_g, const float* lse_g,
                             float* o_out, float* lse_out, uint32_t* status, cudaStream_t st);
cudaError_t launch_decode_attn(int B, int T, int H, const void* q, const uint8_t* codes,
                               const uint8_t* scales, int64_t n_stride, const int32_t* idx, int K,
                               const void* swa, int64_t s_stride, const int32_t* win_start,
                               const int32_t* win_len, int n_win, float scale_log2, float* o,
                               float* lse, int nsplit, float* xchg, uint32_t* status, cudaStream_t st);
cudaError_t launch_ced_project(const void* h, int64_t rows, int d_model, const void* w_kv,
                               const void* w_z, int n_layers, uint8_t* codes, uint8_t* scales,
                               void* z_out, uint32_t* status, cudaStream_t st);
cudaError_t launch_memset_u32(uint32_t* p, size_t n, cudaStream_t st);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

// Order-preserving map of fp32 to uint32 (no NaN); key 0 is never produced. The scoring
// kernels leave each query's min / max score as keys for the selection.
__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// E4M3 code of a non-negative fp32 value, round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

// fp32 value of an E4M3 code (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  uint16_t c = (uint16_t)(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// fp16x2 pair of an E4M3 code placed in both halves (exact).
__device__ __forceinline__ uint32_t e4m3_to_h2(uint32_t code) {
  uint32_t h2;
  uint16_t c = (uint16_t)((code & 0xFFu) * 0x0101u);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return h2;
}

// Eight E2M1 codes (one per nibble, element 0 in the low nibble) from 8 fp32
// values, round to nearest even, saturating at +-6, with -0 stored as +0.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  uint32_t mag = out & 0x77777777u;
  uint32_t nz = (mag + 0x77777777u) & 0x88888888u;  // bit 3 set where magnitude != 0
  return mag | (out & nz);
}

// Four E2M1 codes (low 16 bits, element 0 lowest nibble) -> four fp16 values (2 regs).
__device__ __forceinline__ void e2m1x4_to_h2x2(uint32_t codes16, uint32_t& lo, uint32_t& hi) {
  uint16_t c = (uint16_t)codes16;
  asm("{\n\t.reg .b8 t0, t1;\n\tmov.b16 {t0, t1}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, t0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, t1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "h"(c));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
  int n = valid ? 4 : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D += A * B, m16n8k16, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Convert two bf16 (packed) to fp16x2 (exact for |x| in fp16 normal range).
__device__ __forceinline__ uint32_t bf16x2_to_h2(uint32_t v) {
  return pack_h2(bf16_lo(v), bf16_hi(v));
}
// mag holds, in each 16-bit half, the largest bf16 magnitude bits (value & 0x7FFF) seen:
// true when one of them is above 65280 (0x477F, the largest bf16 value that fp16 holds),
// i.e. an input that is outside the fp16 range or not finite (inf / NaN sort above).
__device__ __forceinline__ bool bf16_mag_beyond_fp16(uint32_t mag) {
  return (mag & 0xFFFFu) > 0x477Fu || (mag >> 16) > 0x477Fu;
}

// Quantise one 16-value block. Returns the 8 code bytes (as two u32) and the
// E4M3 scale code.
__device__ __forceinline__ void quant_block16(const float* v, uint32_t& lo, uint32_t& hi,
                                              uint32_t& scode) {
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(v[k]));
  scode = e4m3_rn_sat(__fdiv_rn(amax, 6.0f));
  float s = e4m3_to_f32(scode);
  if (s == 0.f) {
    lo = hi = 0u;
    return;
  }
  float r[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) r[k] = __fdiv_rn(v[k], s);
  lo = e2m1x8(r);
  hi = e2m1x8(r + 8);
}

// ---- mbarrier and bulk-copy helpers (shared by the TMA-fed kernels)
// Bound on one mbarrier wait: wall time (the global nanosecond timer), checked
// every few hundred polls, so a stalled pipeline turns into an error status
// within about a second instead of spinning.
constexpr uint64_t kMbarWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t a, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(a), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the completion of the phase with the given parity.
__device__ __forceinline__ bool mbar_wait(uint32_t a, uint32_t parity, uint64_t limit_ns = kMbarWaitNs) {
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if (i > 64) __nanosleep(64);
    if ((i & 255) == 0 && global_ns() - t0 > limit_ns) return false;
  }
}

// Requests into L2 (no data returned): `bytes` from a 16-byte aligned address (a
// multiple of 16), or the line holding one address.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}

// ---- tcgen05 helpers (5th-generation tensor cores, accumulators in TMEM)
// Shared-memory matrix descriptor, 128-byte swizzle. K-major operand: rows of
// 128 bytes (64 16-bit elements) in 8-row groups 1024 bytes apart (SBO); the
// leading offset is unused. The start may move by 32 bytes per 16-element
// k-step inside the swizzle span.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1u << 16;              // leading byte offset (unused with 128B swizzle, K-major)
  d |= (uint64_t)(1024u >> 4) << 32;    // stride byte offset: next 8-row group
  d |= (uint64_t)1u << 46;              // descriptor version
  d |= (uint64_t)2u << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   mbar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// MN-major operand with the 128-byte swizzle: atoms of 64 MN-contiguous 16-bit
// elements x 8 K-rows (1024 bytes); lbo = byte stride between atoms along MN,
// sbo = byte stride between 8-row groups along K.
__device__ __forceinline__ uint64_t umma_desc_sw128_mn(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate; a_fmt/b_fmt 0 = fp16, 1 = bf16;
// a_mn/b_mn 1 = MN-major operand.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_fmt, int b_fmt, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_fmt << 7) | ((uint32_t)b_fmt << 10) | ((uint32_t)a_mn << 15) |
         ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

#endif  // __CUDACC__

}  // namespace csa2
