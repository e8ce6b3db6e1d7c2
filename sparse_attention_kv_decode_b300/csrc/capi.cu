// C ABI of libcsa2: host-side validation, workspace checks and dispatch.
// Every entry point validates on the host and launches nothing on a failed
// check; kernels are enqueued on the caller's stream and nothing is allocated.
#include <cudaTypedefs.h>

#include <mutex>

#include "csa2_internal.cuh"

namespace csa2 {

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  std::lock_guard<std::mutex> lk(mu);
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

cudaError_t set_attr_once(int slot, const void* fn, cudaFuncAttribute attr, int value) {
  static std::mutex mu;
  static bool done[64][32] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || slot < 0 || slot >= 32) return cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev][slot]) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, attr, value);
  if (e == cudaSuccess) done[dev][slot] = true;
  return e;
}

// cuTensorMapEncodeTiled is reached through the runtime's driver entry point,
// so the library does not link against the driver library.
static PFN_cuTensorMapEncodeTiled_v12000 encode_tiled_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode_tensor_map_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                               uint32_t box_inner, uint32_t box_outer) {
  auto encode = encode_tiled_fn();
  if (encode == nullptr) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                      dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int attn_splits(int64_t Q, int K, int W, int n_sm) {
  if (Q <= 0) return 1;
  int64_t s = n_sm / Q;                  // at most one wave of one-CTA-per-SM blocks
  // at least one 128-key tile per split; the window's tiles go to the last split
  int64_t max_by_k = (K + 127) / 128 + (W > 0 ? (W + 127) / 128 : 0);
  if (s > max_by_k) s = max_by_k;
  if (s > kMaxSplits) s = kMaxSplits;
  int p = 1;                             // splits form one cluster: a power of two
  while (2 * p <= s) p *= 2;
  return p;
}

}  // namespace csa2

using namespace csa2;

static inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

#define CHECK_ARG(cond)                       \
  do {                                        \
    if (!(cond)) return CSA2_ERR_INVALID_ARG; \
  } while (0)

static thread_local const char* g_last_cuda_error = "no error";

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return CSA2_OK;
  g_last_cuda_error = cudaGetErrorString(e);
  return CSA2_ERR_CUDA;
}

// Scratch of csa2_index_topk_noalloc: the 256-byte status header, the score
// range words of up to 8192 queries (64 KiB), then room for 2^21 fp32 indexer
// scores (8 MiB), e.g. 32 queries over 65,536 entries or 4 queries over 262,144.
// It is part of the module image (zero at load).
constexpr size_t kStaticScratchBytes = kWsHeader + 65536 + (size_t(1) << 23);
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch for the current device. Outside a stream
// capture it is looked up on every call (so a context torn down and created again
// since the last call gets its own address); inside a capture, where the lookup
// could load the module, the address of the last call outside one is used, and a
// capture before any such call is refused.
static int static_scratch(cudaStream_t st, void** out) {
  static std::mutex mu;
  static void* cache[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= 64) return CSA2_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) return cuda_status(e);
  std::lock_guard<std::mutex> lk(mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_status(e);
    if (p == nullptr) return CSA2_ERR_CUDA;
    cache[dev] = p;
  } else if (cache[dev] == nullptr) {
    return CSA2_ERR_UNSUPPORTED;
  }
  *out = cache[dev];
  return CSA2_OK;
}

extern "C" {

int csa2_version(void) { return 200; }

const char* csa2_last_cuda_error(void) { return g_last_cuda_error; }

const char* csa2_status_string(int s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSA2_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_TIMEOUT: return "device-side wait or refinement limit reached";
    case CSA2_ERR_DEVICE_CHECK: return "device-side bounds check fired";
    default: return "unknown status";
  }
}

// The attention's split exchange (few queries, clusters of 2 or 4 CTAs): per query
// nsplit x 512 dims x 64 heads fp32 partial outputs, at the end of the workspace.
constexpr size_t kXchgPerSplit = (size_t)512 * 64 * 4;
constexpr int64_t kXchgMaxQ = 128;   // clusters of more than one CTA need Q <= SMs / 2
static size_t xchg_bytes(int64_t Q) { return Q <= kXchgMaxQ ? (size_t)Q * 4 * kXchgPerSplit : 0; }
static size_t index_ws_bytes(int64_t Q, int64_t n_max, int K) {
  return kWsHeader + range_bytes(Q) + scores_bytes(Q, n_max) + pool_bytes(Q, K);
}
// The exchange buffer of an attention call with nsplit CTAs per query, placed at the end
// of the workspace past its first `front` bytes; nullptr when the call needs none or the
// workspace is too small for it (the splits then merge through distributed shared memory).
static float* attn_xchg(void* ws, size_t ws_bytes, size_t front, int64_t Q, int nsplit) {
  if (nsplit < 2 || nsplit > 4 || ws == nullptr) return nullptr;
  const size_t need = (size_t)Q * nsplit * kXchgPerSplit;
  if (ws_bytes < front + need) return nullptr;
  const size_t at = (ws_bytes - need) & ~(size_t)255;
  return at >= front ? reinterpret_cast<float*>(static_cast<char*>(ws) + at) : nullptr;
}

size_t csa2_workspace_bytes(int B, int T, int H, int64_t n_max, int K) {
  if (B < 0 || T < 0 || H < 0 || n_max < 0 || K < 0) return 0;
  (void)H;
  const int64_t Q = (int64_t)B * T;
  return index_ws_bytes(Q, n_max, K) + xchg_bytes(Q);
}

int csa2_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  CHECK_ARG(ws != nullptr && ws_bytes >= kWsHeader && aligned(ws, 256));
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream));
}

int csa2_read_device_status(void* ws, void* stream, uint32_t* flags) {
  CHECK_ARG(ws != nullptr);
  uint32_t v = 0;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&v, ws, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws, 0, 4, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_status(e);
  if (flags) *flags = v;
  if (v == 0) return CSA2_OK;
  if ((v & ~(CSA2_DEV_TOPK_LEVELS | CSA2_DEV_PIPELINE_TIMEOUT)) == 0) return CSA2_ERR_TIMEOUT;
  return CSA2_ERR_DEVICE_CHECK;
}

int csa2_encode_kv(const void* h, int h_dtype, int64_t rows, int d_model, const void* w_kv,
                   const void* w_z, int n_layers, uint8_t* kv_codes, uint8_t* kv_scales,
                   void* z_out, void* ws, size_t ws_bytes, void* stream) {
  CHECK_ARG(rows >= 0 && n_layers >= 1);
  CHECK_ARG(h_dtype == CSA2_F32 || h_dtype == CSA2_BF16);
  cudaStream_t st = (cudaStream_t)stream;
  if (w_kv == nullptr && w_z == nullptr) {
    CHECK_ARG(d_model == CSA2_D_KV && n_layers == 1 && z_out == nullptr);
    if (rows == 0) return CSA2_OK;
    CHECK_ARG(h && kv_codes && kv_scales);
    CHECK_ARG(aligned(h, 16) && aligned(kv_codes, 8));
    return cuda_status(launch_encode_quant(h, h_dtype, rows, kv_codes, kv_scales, st));
  }
  CHECK_ARG(w_kv && w_z && z_out);
  CHECK_ARG(h_dtype == CSA2_BF16);
  CHECK_ARG(d_model >= 64 && d_model % 64 == 0);
  if (rows == 0) return CSA2_OK;
  CHECK_ARG(h && kv_codes && kv_scales);
  CHECK_ARG(aligned(h, 16) && aligned(w_kv, 16) && aligned(w_z, 16) && aligned(kv_codes, 16) &&
            aligned(kv_scales, 4) && aligned(z_out, 16));
  if (rows > ((int64_t)1 << 30)) return CSA2_ERR_UNSUPPORTED;
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  CHECK_ARG(aligned(ws, 256));
  if (ws_bytes < kWsHeader) return CSA2_ERR_WORKSPACE;
  return cuda_status(launch_ced_project(h, rows, d_model, w_kv, w_z, n_layers, kv_codes, kv_scales,
                                        z_out, static_cast<uint32_t*>(ws), st));
}

int csa2_check_bounded_wait(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream) {
  CHECK_ARG(limit_ns >= 1000 && limit_ns <= (int64_t)kMbarWaitNs);
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  CHECK_ARG(aligned(ws, 256));
  if (ws_bytes < kWsHeader) return CSA2_ERR_WORKSPACE;
  return cuda_status(launch_wait_check((uint64_t)limit_ns, static_cast<uint32_t*>(ws), (cudaStream_t)stream));
}

int csa2_cache_append(int B, int32_t* n_tokens, int advance, int ratio, const void* swa_row, void* swa_kv,
                      int64_t s_stride, int n_win, const void* entry_kv, int entry_dtype, const void* entry_z,
                      uint8_t* kv_codes, uint8_t* kv_scales, void* z, int64_t n_stride, int32_t* n_visible,
                      int32_t* win_start, int32_t* win_len, void* ws, size_t ws_bytes, void* stream) {
  CHECK_ARG(B >= 0 && ratio >= 1 && n_stride >= 0 && s_stride >= 0 && n_win >= 0);
  CHECK_ARG((win_start == nullptr) == (win_len == nullptr));
  if (swa_row != nullptr || win_start != nullptr) CHECK_ARG(n_win >= 1);
  if (swa_row != nullptr) {
    CHECK_ARG(swa_kv != nullptr && s_stride >= 2 * (int64_t)n_win);
    CHECK_ARG(aligned(swa_row, 16) && aligned(swa_kv, 16));
  }
  if (entry_kv != nullptr) {
    CHECK_ARG(entry_dtype == CSA2_F32 || entry_dtype == CSA2_BF16);
    CHECK_ARG(kv_codes != nullptr && kv_scales != nullptr);
    CHECK_ARG(aligned(entry_kv, 16) && aligned(kv_codes, 8));
  }
  if (entry_z != nullptr) CHECK_ARG(z != nullptr && aligned(entry_z, 16) && aligned(z, 16));
  if (B == 0) return CSA2_OK;
  CHECK_ARG(n_tokens != nullptr);
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  CHECK_ARG(aligned(ws, 256));
  if (ws_bytes < kWsHeader) return CSA2_ERR_WORKSPACE;
  return cuda_status(launch_cache_append(B, n_tokens, advance, ratio, swa_row, swa_kv, s_stride, n_win, entry_kv,
                                         entry_dtype, entry_z, kv_codes, kv_scales, z, n_stride, n_visible,
                                         win_start, win_len, static_cast<uint32_t*>(ws),
                                         (cudaStream_t)stream));
}

}  // extern "C"

// Argument checks of csa2_decode_attention (CSA2_OK also for an empty batch).
static int check_decode_attention(int B, int T, int H, const void* q, const uint8_t* kv_codes,
                                  const uint8_t* kv_scales, int64_t n_stride, const int32_t* idx,
                                  int K, const void* swa_kv, int64_t s_stride,
                                  const int32_t* win_start, const int32_t* win_len, int n_win,
                                  int d_v, float softmax_scale, float* o, float* lse, void* ws,
                                  size_t ws_bytes) {
  CHECK_ARG(B >= 0 && T >= 0 && H >= 1 && K >= 1 && n_stride >= 0 && s_stride >= 0 && n_win >= 0);
  CHECK_ARG(softmax_scale == softmax_scale);
  if (H % 16 != 0 || H > 64 || d_v != CSA2_D_LATENT || K > kMaxK || n_win > kMaxWin)
    return CSA2_ERR_UNSUPPORTED;
  const int64_t Q = (int64_t)B * T;
  if (Q == 0) return CSA2_OK;
  CHECK_ARG(q && idx && o && win_start && win_len);
  CHECK_ARG(n_stride == 0 || (kv_codes && kv_scales));
  CHECK_ARG(s_stride == 0 || swa_kv != nullptr);
  CHECK_ARG(aligned(q, 16) && aligned(kv_codes, 16) && aligned(kv_scales, 4) && aligned(idx, 4) &&
            aligned(swa_kv, 16) && aligned(win_start, 4) && aligned(win_len, 4) && aligned(o, 16) &&
            aligned(lse, 4));
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  CHECK_ARG(aligned(ws, 256));
  if (ws_bytes < kWsHeader) return CSA2_ERR_WORKSPACE;
  return CSA2_OK;
}

// front: the workspace bytes in use by the call's other parts (the split exchange goes
// past them)
static int decode_attention_launch(int B, int T, int H, const void* q, const uint8_t* kv_codes,
                                   const uint8_t* kv_scales, int64_t n_stride, const int32_t* idx,
                                   int K, const void* swa_kv, int64_t s_stride,
                                   const int32_t* win_start, const int32_t* win_len, int n_win,
                                   float softmax_scale, float* o, float* lse, void* ws,
                                   size_t ws_bytes, size_t front, void* stream) {
  const int64_t Q = (int64_t)B * T;
  const int nsplit = attn_splits(Q, K, n_win, device_sm_count());
  uint32_t* status = static_cast<uint32_t*>(ws);
  const float scale_log2 = softmax_scale * 1.4426950408889634074f;
  return cuda_status(launch_decode_attn(B, T, H, q, kv_codes, kv_scales, n_stride, idx, K, swa_kv,
                                        s_stride, win_start, win_len, n_win, scale_log2, o, lse,
                                        nsplit, attn_xchg(ws, ws_bytes, front, Q, nsplit), status,
                                        (cudaStream_t)stream));
}

// csa2_index_topk; pf_codes / pf_scales (nullable) name the FP4 cache whose rows of the
// selected entries the selection requests into L2
static int index_topk_impl(int mode, int B, int T, int H_I, const void* q_idx, const float* w_idx,
                           const void* z, int64_t n_stride, const int32_t* n_visible, int K,
                           const int32_t* prev_idx, int32_t* out_idx, float* out_scores, void* ws,
                           size_t ws_bytes, void* stream, const uint8_t* pf_codes,
                           const uint8_t* pf_scales) {
  CHECK_ARG(mode == CSA2_MODE_FULL || mode == CSA2_MODE_REINDEX || mode == CSA2_MODE_REUSE ||
            mode == CSA2_MODE_REINDEX_POOL);
  CHECK_ARG(B >= 0 && T >= 0 && K >= 1);
  if (K > kMaxK) return CSA2_ERR_UNSUPPORTED;
  const int64_t Q = (int64_t)B * T;
  cudaStream_t st = (cudaStream_t)stream;
  if (mode == CSA2_MODE_REUSE) {
    CHECK_ARG(prev_idx != nullptr);
    if (Q == 0) return CSA2_OK;
    CHECK_ARG(out_idx != nullptr);
    return cuda_status(launch_copy_idx(prev_idx, out_idx, Q * K, st));
  }
  CHECK_ARG(H_I >= 1 && n_stride >= 0);
  if (H_I > 16 || n_stride > kMaxNStride) return CSA2_ERR_UNSUPPORTED;
  if (Q == 0) return CSA2_OK;
  CHECK_ARG(q_idx && w_idx && n_visible && out_idx);
  CHECK_ARG(n_stride == 0 || z != nullptr);
  CHECK_ARG(aligned(q_idx, 16) && aligned(z, 16) && aligned(w_idx, 4) && aligned(out_idx, 4) &&
            aligned(n_visible, 4) && aligned(out_scores, 4) && aligned(prev_idx, 4));
  // REINDEX_POOL searches only the candidate pool of prev_idx (the first FULL layer's selection)
  const bool pooled = mode == CSA2_MODE_REINDEX_POOL;
  CHECK_ARG(!pooled || prev_idx != nullptr);
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  CHECK_ARG(aligned(ws, 256));
  // REINDEX_POOL scores at most K blocks x 8 positions per query, and no more than the
  // (8-aligned) cache rows: its score rows are that long, not n_stride
  const int64_t n8 = (n_stride + 7) / 8 * 8;
  const int64_t pcap = (int64_t)8 * K < n8 ? (int64_t)8 * K : n8;
  const int64_t pstride = score_pad(pcap);
  const size_t after_scores =
      kWsHeader + range_bytes(Q) + (pooled ? (size_t)Q * (size_t)pstride * 4 : scores_bytes(Q, n_stride));
  if (ws_bytes < after_scores + (pooled ? pool_bytes(Q, K) : 0)) return CSA2_ERR_WORKSPACE;
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  uint32_t* range = reinterpret_cast<uint32_t*>(wsb + kWsHeader);
  float* scores = reinterpret_cast<float*>(wsb + kWsHeader + range_bytes(Q));
  uint32_t* status = reinterpret_cast<uint32_t*>(wsb);
  if (pooled) {
    int32_t* blocks = reinterpret_cast<int32_t*>(wsb + after_scores);
    int32_t* pool_nv = reinterpret_cast<int32_t*>(wsb + after_scores + ((size_t)Q * K * 4 + 255) / 256 * 256);
    cudaError_t e = launch_pool_build(prev_idx, (int)Q, K, n_visible, n_stride, blocks, pool_nv, status, st);
    if (e == cudaSuccess)
      e = launch_index_score(q_idx, w_idx, z, n_stride, n_visible, B, T, H_I, scores, pstride, range,
                             status, st, blocks, pool_nv, K);
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(launch_topk_select(scores, pstride, pool_nv, (int)Q, pcap, K, range, out_idx,
                                          out_scores, status, st, pf_codes, pf_scales, T, n_stride,
                                          blocks, K));
  }
  const int64_t stride = score_pad(n_stride);
  // keys x (token, head) products on the tensor cores: N = 256 columns with many query
  // tokens per sequence (prefill), N = 16 with few (decode)
  cudaError_t e;
  if (index_gemm_applies(T, H_I))
    e = launch_index_gemm(q_idx, w_idx, z, n_stride, n_visible, B, T, H_I, scores, stride, range, status, st);
  else if (index_stream_applies(B, T, H_I))
    e = launch_index_stream(q_idx, w_idx, z, n_stride, n_visible, B, T, H_I, scores, stride, range, status, st);
  else
    e = launch_index_score(q_idx, w_idx, z, n_stride, n_visible, B, T, H_I, scores, stride, range, status, st);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_topk_select(scores, stride, n_visible, (int)Q, n_stride, K, range,
                                        out_idx, out_scores, status, st, pf_codes, pf_scales, T));
}

extern "C" {

int csa2_index_topk(int mode, int B, int T, int H_I, const void* q_idx, const float* w_idx,
                    const void* z, int64_t n_stride, const int32_t* n_visible, int K,
                    const int32_t* prev_idx, int32_t* out_idx, float* out_scores, void* ws,
                    size_t ws_bytes, void* stream) {
  return index_topk_impl(mode, B, T, H_I, q_idx, w_idx, z, n_stride, n_visible, K, prev_idx,
                         out_idx, out_scores, ws, ws_bytes, stream, nullptr, nullptr);
}

int csa2_index_topk_prefetch(int mode, int B, int T, int H_I, const void* q_idx, const float* w_idx,
                             const void* z, int64_t n_stride, const int32_t* n_visible, int K,
                             const int32_t* prev_idx, int32_t* out_idx, float* out_scores,
                             const uint8_t* kv_codes, const uint8_t* kv_scales, void* ws,
                             size_t ws_bytes, void* stream) {
  CHECK_ARG(mode == CSA2_MODE_REUSE || n_stride == 0 || (kv_codes && kv_scales));
  CHECK_ARG(aligned(kv_codes, 16));
  return index_topk_impl(mode, B, T, H_I, q_idx, w_idx, z, n_stride, n_visible, K, prev_idx,
                         out_idx, out_scores, ws, ws_bytes, stream, kv_codes, kv_scales);
}

int csa2_index_topk_noalloc(int mode, int B, int T, int H_I, const void* q_idx,
                            const float* w_idx, const void* z, int64_t n_stride,
                            const int32_t* n_visible, int K, const int32_t* prev_idx,
                            int32_t* out_idx, float* out_scores, void* stream) {
  // REUSE touches no scratch; the other modes run csa2_index_topk's own validation
  // and kernels on the static scratch, which rejects more than 2^21 scores with
  // CSA2_ERR_WORKSPACE before launching anything
  void* scratch = nullptr;
  if (mode != CSA2_MODE_REUSE) {
    const int s = static_scratch((cudaStream_t)stream, &scratch);
    if (s != CSA2_OK) return s;
  }
  return csa2_index_topk(mode, B, T, H_I, q_idx, w_idx, z, n_stride, n_visible, K, prev_idx,
                         out_idx, out_scores, scratch, scratch ? kStaticScratchBytes : 0, stream);
}

int csa2_sparse_decode(int B, int T, int H, const void* q, const uint8_t* kv_codes,
                       const uint8_t* kv_scales, int64_t n_stride, const int32_t* idx, int K,
                       int d_v, float softmax_scale, float* o_g, float* lse_g, void* ws,
                       size_t ws_bytes, void* stream) {
  CHECK_ARG(B >= 0 && T >= 0 && H >= 1 && K >= 1 && n_stride >= 0);
  CHECK_ARG(softmax_scale == softmax_scale);  // not NaN
  if (H % 16 != 0 || H > 64 || d_v != CSA2_D_LATENT || K > kMaxK) return CSA2_ERR_UNSUPPORTED;
  const int64_t Q = (int64_t)B * T;
  if (Q == 0) return CSA2_OK;
  CHECK_ARG(q && idx && o_g && lse_g);
  CHECK_ARG(n_stride == 0 || (kv_codes && kv_scales));
  CHECK_ARG(aligned(q, 16) && aligned(kv_codes, 16) && aligned(kv_scales, 4) &&
            aligned(o_g, 16) && aligned(lse_g, 4) && aligned(idx, 4));
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  CHECK_ARG(aligned(ws, 256));
  const int nsplit = attn_splits(Q, K, 0, device_sm_count());
  if (ws_bytes < kWsHeader) return CSA2_ERR_WORKSPACE;
  uint32_t* status = static_cast<uint32_t*>(ws);
  const float scale_log2 = softmax_scale * 1.4426950408889634074f;
  return cuda_status(launch_sparse_attn(B, T, H, q, kv_codes, kv_scales, n_stride, idx, K,
                                        scale_log2, o_g, lse_g, nsplit,
                                        attn_xchg(ws, ws_bytes, kWsHeader + range_bytes(Q), Q, nsplit), status,
                                        (cudaStream_t)stream));
}

int csa2_swa_merge(int B, int T, int H, const void* q, const void* swa_kv, int64_t s_stride,
                   const int32_t* win_start, const int32_t* win_len, int n_win, int d_v,
                   float softmax_scale, const float* o_g, const float* lse_g, float* o_out,
                   float* lse_out, void* ws, size_t ws_bytes, void* stream) {
  CHECK_ARG(B >= 0 && T >= 0 && H >= 1 && s_stride >= 0 && n_win >= 0);
  CHECK_ARG(softmax_scale == softmax_scale);
  if (H % 16 != 0 || H > 64 || d_v != CSA2_D_LATENT || n_win > kMaxWin) return CSA2_ERR_UNSUPPORTED;
  const int64_t Q = (int64_t)B * T;
  if (Q == 0) return CSA2_OK;
  CHECK_ARG(q && win_start && win_len && o_g && lse_g && o_out);
  CHECK_ARG(s_stride == 0 || swa_kv != nullptr);
  CHECK_ARG(aligned(q, 16) && aligned(swa_kv, 16) && aligned(o_g, 16) && aligned(lse_g, 4) &&
            aligned(o_out, 16) && aligned(lse_out, 4) && aligned(win_start, 4) &&
            aligned(win_len, 4));
  if (ws == nullptr) return CSA2_ERR_WORKSPACE;
  CHECK_ARG(aligned(ws, 256));
  if (ws_bytes < kWsHeader) return CSA2_ERR_WORKSPACE;
  uint32_t* status = static_cast<uint32_t*>(ws);
  const float scale_log2 = softmax_scale * 1.4426950408889634074f;
  return cuda_status(launch_swa_merge(B, T, H, q, swa_kv, s_stride, win_start, win_len, n_win,
                                      scale_log2, o_g, lse_g, o_out, lse_out, status,
                                      (cudaStream_t)stream));
}

int csa2_decode_attention(int B, int T, int H, const void* q, const uint8_t* kv_codes,
                          const uint8_t* kv_scales, int64_t n_stride, const int32_t* idx, int K,
                          const void* swa_kv, int64_t s_stride, const int32_t* win_start,
                          const int32_t* win_len, int n_win, int d_v, float softmax_scale, float* o,
                          float* lse, void* ws, size_t ws_bytes, void* stream) {
  const int s = check_decode_attention(B, T, H, q, kv_codes, kv_scales, n_stride, idx, K, swa_kv,
                                       s_stride, win_start, win_len, n_win, d_v, softmax_scale, o,
                                       lse, ws, ws_bytes);
  if (s != CSA2_OK || (int64_t)B * T == 0) return s;
  return decode_attention_launch(B, T, H, q, kv_codes, kv_scales, n_stride, idx, K, swa_kv, s_stride,
                                 win_start, win_len, n_win, softmax_scale, o, lse, ws, ws_bytes,
                                 kWsHeader + range_bytes((int64_t)B * T), stream);
}

int csa2_decode_layer(int mode, int B, int T, int H, int H_I, const void* q, const void* q_idx,
                      const float* w_idx, const void* z, const uint8_t* kv_codes,
                      const uint8_t* kv_scales, int64_t n_stride, const int32_t* n_visible, int K,
                      const int32_t* prev_idx, int32_t* out_idx, const void* swa_kv,
                      int64_t s_stride, const int32_t* win_start, const int32_t* win_len,
                      int n_win, int d_v, float softmax_scale, float* o, float* lse, void* ws,
                      size_t ws_bytes, void* stream) {
  // both halves are validated before either launches
  int s = check_decode_attention(B, T, H, q, kv_codes, kv_scales, n_stride, out_idx, K, swa_kv,
                                 s_stride, win_start, win_len, n_win, d_v, softmax_scale, o, lse,
                                 ws, ws_bytes);
  if (s != CSA2_OK) return s;
  // the selection does not request the selected entries into L2 here: the attention's own
  // requests (and its register gather) find them soon enough, and 25 MB of requests queued
  // at the selection's end delayed the attention's first tile (measured: 1.9 us per layer)
  s = index_topk_impl(mode, B, T, H_I, q_idx, w_idx, z, n_stride, n_visible, K, prev_idx, out_idx,
                      nullptr, ws, ws_bytes, stream, nullptr, nullptr);
  if (s != CSA2_OK || (int64_t)B * T == 0) return s;
  return decode_attention_launch(B, T, H, q, kv_codes, kv_scales, n_stride, out_idx, K, swa_kv,
                                 s_stride, win_start, win_len, n_win, softmax_scale, o, lse, ws,
                                 ws_bytes, kWsHeader + range_bytes((int64_t)B * T), stream);
}

}  // extern "C"
