/*
 * csa2.h - C ABI of the CSA2 FP4 sparse-decode library (libcsa2.so, sm_103a).
 *
 * Decode-time global attention of Compressed Sparse Attention 2 over an FP4
 * compressed KV cache, and the CED projection that fills that cache, as
 * described in "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
 * Compression" (picx.dev summary, Methodology / Architecture Components:
 * 1. CED, Eq. (1); 2. CSA2 layer modes; 5. FP4 Main KV Cache; and the blog
 * repost's description of sparse attention combined with a sliding window).
 *
 * Conventions shared by every entry point
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise. The
 *    caller owns all buffers; the library never allocates or frees memory and
 *    keeps no state beyond per-device kernel attributes set on first use.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Calls only enqueue work: they are asynchronous and stream-ordered.
 *    Calls are thread-safe.
 *  - Arguments are validated on the host before anything is launched; a failed
 *    check returns a non-zero csa2_status and launches nothing. A launch error
 *    returns CSA2_ERR_CUDA.
 *  - Problems only the device can see (an index outside the cache, a window
 *    outside the store) never trap: the offending element is skipped and a bit
 *    is set in the status word at the start of the workspace; read it with
 *    csa2_read_device_status.
 *  - bf16 tensors are IEEE bfloat16 bit patterns (uint16). Shapes are given
 *    row-major, innermost last.
 *  - FP4 main-KV layout: an entry of 576 channels (512 latent + 64 rope) is
 *    288 bytes of E2M1 codes (channel 2i in the low nibble of byte i, 2i+1 in
 *    the high nibble; sign in bit 3 of the nibble) and 36 bytes of E4M3 scales
 *    (scale j covers channels 16j..16j+15). dequant = e2m1(code) * e4m3(scale).
 *    Entries are rows of CSA2_ENTRY_BYTES (384) bytes: every kv_codes /
 *    kv_scales argument below is a pointer to the 288 code bytes / the 36 scale
 *    bytes of the first entry, and entry n of either is CSA2_ENTRY_BYTES * n
 *    bytes further on. The library's own layout (the one that saves DRAM
 *    traffic) is one record per entry: kv_scales = kv_codes + 288, then 60
 *    bytes of padding the library never reads or writes; with 128-byte aligned
 *    records a gathered entry is exactly three 128-byte L2 lines (324 bytes
 *    used of 384). Separate code and scale arrays with the same 384-byte row
 *    stride work too (and cost more DRAM traffic).
 */
#ifndef CSA2_H_
#define CSA2_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or mode   */
  CSA2_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels cover */
  CSA2_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required   */
  CSA2_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed         */
  CSA2_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up            */
  CSA2_ERR_DEVICE_CHECK = 6   /* a device-side bounds check fired              */
} csa2_status;

typedef enum { CSA2_MODE_FULL = 0, CSA2_MODE_REINDEX = 1, CSA2_MODE_REUSE = 2,
               CSA2_MODE_REINDEX_POOL = 3 } csa2_mode;
typedef enum { CSA2_F32 = 0, CSA2_BF16 = 1 } csa2_dtype;

/* Fixed dimensions of the format. */
#define CSA2_D_KV 576        /* latent 512 + rope 64 channels per entry      */
#define CSA2_D_LATENT 512
#define CSA2_D_IDX 64        /* indexer key / query width                    */
#define CSA2_CODE_BYTES 288  /* E2M1 bytes per entry                         */
#define CSA2_SCALE_BYTES 36  /* E4M3 scale bytes per entry                   */
#define CSA2_ENTRY_BYTES 384 /* row stride of kv_codes and kv_scales (bytes)  */

/* Device status bits (csa2_read_device_status). */
#define CSA2_DEV_BAD_INDEX 0x1u   /* sparse_decode saw idx >= n_stride or < -1 */
#define CSA2_DEV_BAD_WINDOW 0x2u  /* swa_merge window outside [0, s_stride)    */
#define CSA2_DEV_TOPK_LEVELS 0x4u /* top-K refinement did not settle           */
#define CSA2_DEV_PIPELINE_TIMEOUT 0x8u /* a bounded mbarrier wait gave up       */
#define CSA2_DEV_RANGE 0x10u      /* a bf16 query / window value outside fp16 range */

/*
 * csa2_encode_kv - write the FP4 main KV cache.
 *
 * (a) Quantise-only (w_kv == NULL and w_z == NULL): h is [rows][576] in
 *     h_dtype (fp32 or bf16), d_model must be 576, n_layers must be 1 and
 *     z_out must be NULL. Writes kv_codes and kv_scales rows 0..rows-1.
 *     Per 16-channel block: s = E4M3_RNE_satfinite(fl32(amax / 6)); each code
 *     = E2M1_RNE_satfinite(fl32(x / s)); a zero scale stores zero codes and a
 *     value rounding to zero stores +0. (FP4 Main KV Cache, picx.dev summary.)
 * (b) CED projection, Eq. (1): C_l = H W_l^KV and Z_l = H W_l^Z for
 *     l = 0..n_layers-1. h is bf16 [rows][d_model]; w_kv is bf16
 *     [n_layers][576][d_model] and w_z bf16 [n_layers][64][d_model] (row c
 *     holds the weights of output channel c, i.e. W^T). Writes kv_codes /
 *     kv_scales rows l*rows .. l*rows+rows-1 for layer l (C_l quantised
 *     as in (a) from its fp32 value) and z_out bf16 [n_layers][rows][64]
 *     (round to nearest even). Requires h_dtype == CSA2_BF16,
 *     d_model % 64 == 0, rows <= 2^30, 16-byte aligned h/w_kv/w_z/kv_codes/
 *     z_out. The fp32 product is accumulated by the tensor cores, so a block
 *     whose exact product sits within the accumulation error of a rounding
 *     boundary may round either way. ws must hold at least 256 bytes (the
 *     status word); a bounded device wait that gives up sets
 *     CSA2_DEV_PIPELINE_TIMEOUT there.
 * (a) ignores ws (pass NULL, 0).
 */
CSA2_API int csa2_encode_kv(const void* h, int h_dtype, int64_t rows, int d_model,
                   const void* w_kv, const void* w_z, int n_layers,
                   uint8_t* kv_codes, uint8_t* kv_scales, void* z_out,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_index_topk - per-query top-K entry selection of a CSA2 layer.
 *
 * FULL / REINDEX: scores every visible entry n < n_visible[b*T+t] with
 *   I[n] = sum_h w_idx[h] * max(0, q_idx[h] . z[n])   (h < H_I)
 * and writes the K best to out_idx [B][T][K] int32, ascending by index, with
 * equal scores going to the lower index and -1 padding when fewer than K are
 * visible; out_scores [B][T][K] (nullable) receives their fp32 scores (NaN at
 * padding). The two modes compute the same selection from the layer's own
 * indexer query and keys; they differ in which main KV the caller attends
 * over (CSA2 layer modes, picx.dev summary). The score formula is this
 * library's reading: the pages name the indexer but print no formula.
 * q_idx: bf16 [B][T][H_I][64]; w_idx: fp32 [B][T][H_I]; z: bf16
 * [B][n_stride][64]; n_visible: int32 [B*T], each in [0, n_stride].
 * Limits: 1 <= H_I <= 16, 1 <= K <= 4096, n_stride <= 262144 (1M tokens at 4:1).
 * REUSE: copies prev_idx [B][T][K] to out_idx (nothing to do when they are
 *   the same pointer); q_idx, w_idx, z, n_visible and out_scores are ignored.
 * REINDEX_POOL: REINDEX restricted to the candidate pool of the Hierarchical Sparse
 *   Indexer (picx.dev summary, Methodology / 3): prev_idx [B][T][K] is the first FULL
 *   layer's selection (as written by this call: ascending, -1 padded), and query (b,t)
 *   ranks only the positions of the aligned 8-entry blocks holding one of its entries
 *   (at most 8K positions), below n_visible, under the same rules; the cost no longer
 *   grows with n_stride. A prev_idx that is not ascending or holds an index outside
 *   [-1, n_stride) sets CSA2_DEV_BAD_INDEX. The block reading is this library's
 *   (the page gives "2,048 blocks x 8 positions").
 * ws: at least csa2_workspace_bytes(B, T, *, n_stride, K) bytes, prepared
 * once by csa2_workspace_init (REINDEX_POOL needs only 256 + roundup256(8 B T) +
 * 4 B T P + roundup256(4 B T K) + roundup256(4 B T) bytes, with P =
 * roundup1024(min(8 K, roundup8(n_stride))) pool positions per query).
 */
CSA2_API int csa2_index_topk(int mode, int B, int T, int H_I,
                    const void* q_idx, const float* w_idx,
                    const void* z, int64_t n_stride, const int32_t* n_visible,
                    int K, const int32_t* prev_idx, int32_t* out_idx, float* out_scores,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_index_topk_prefetch - csa2_index_topk whose selection also requests the FP4
 * rows (kv_codes / kv_scales rows [B][n_stride], the cache the
 * attention that follows gathers from) of the entries it selects into L2.
 *
 * Not in the pages: a scheduling aid with the same results as csa2_index_topk;
 * the attention's gathers then find the rows in L2. kv_codes 16-byte aligned;
 * both may be null only in REUSE mode (which prefetches nothing).
 */
CSA2_API int csa2_index_topk_prefetch(int mode, int B, int T, int H_I,
                    const void* q_idx, const float* w_idx,
                    const void* z, int64_t n_stride, const int32_t* n_visible,
                    int K, const int32_t* prev_idx, int32_t* out_idx, float* out_scores,
                    const uint8_t* kv_codes, const uint8_t* kv_scales,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_index_topk_noalloc - csa2_index_topk without a caller workspace.
 *
 * Not part of the method (the pages describe no such call): the same selection
 * as csa2_index_topk (same arguments, kernels and results), with its scratch in
 * a fixed device array inside this library (256 B header + 64 KiB of per-query
 * score ranges + 8 MiB of scores), so the call allocates nothing and needs no
 * workspace. It is for callers that cannot allocate device memory for one: a
 * serving engine that reserves all free device memory for its own KV pool at
 * start-up, or a plug-in that receives tensors from a host framework but no
 * allocator. Every GPU that loads the library holds the array until exit.
 * Limit: with Q = B * T, FULL / REINDEX need 256 B + roundup256(8 Q) + 4 Q *
 *   roundup1024(n_stride) bytes, at most 256 B + 64 KiB + 8 MiB: up to 2^21
 *   padded scores, hence at most 2048 queries (e.g. 32 queries over 65,536
 *   entries). REINDEX_POOL scores only its pool, P = roundup1024(min(8 K,
 *   roundup8(n_stride))) positions per query, and needs 256 B + roundup256(8 Q)
 *   + 4 Q P + roundup256(4 Q K) + roundup256(4 Q) bytes (e.g. 32 queries with
 *   K = 2048 at any n_stride). Larger calls return CSA2_ERR_WORKSPACE and launch
 *   nothing. REUSE has no limit (it uses no scratch).
 * Set-up: every FULL/REINDEX/REINDEX_POOL call made outside a stream capture
 *   looks up the array's address on the current device (cudaGetSymbolAddress,
 *   which may load the module; a failed lookup returns CSA2_ERR_CUDA); a call
 *   inside a capture uses the address found by the last call outside one on
 *   that device, so make one call on each device before capturing (a capture
 *   before any returns CSA2_ERR_UNSUPPORTED).
 * Starting values: the array is zero when the module loads, which is the state
 *   the per-query score-range words must start in; each call leaves them zero
 *   again (the selection is exact from any start, a non-zero leftover only
 *   costs it an extra round). The scores are written before they are read.
 *   Device-check bits (CSA2_DEV_*) are recorded in the array's status word and
 *   are not reported; use csa2_index_topk with a workspace to read them.
 * One scratch per device: calls that may overlap on a device (two streams, two
 *   threads) race on it and must be serialised by the caller.
 */
CSA2_API int csa2_index_topk_noalloc(int mode, int B, int T, int H_I,
                    const void* q_idx, const float* w_idx,
                    const void* z, int64_t n_stride, const int32_t* n_visible,
                    int K, const int32_t* prev_idx, int32_t* out_idx, float* out_scores,
                    void* stream);

/*
 * csa2_sparse_decode - global branch: sparse MQA over the selected FP4 entries.
 *
 * For each query (b, t) and head h < H:
 *   s_j = softmax_scale * q[b,t,h,:] . C[b, idx[b,t,j], :]   (576 channels)
 *   O_g[b,t,h,:] = sum_j softmax(s)_j * C[b, idx_j, 0:d_v],
 *   LSE_g[b,t,h] = log sum_j exp(s_j)  (natural log),
 * over the j with idx >= 0; C is dequantised in registers from kv_codes
 * / kv_scales rows [B][n_stride]. One KV entry is shared by
 * all heads (MQA). An empty selection gives O_g = 0 and LSE_g = -inf.
 * q: bf16 [B][T][H][576]; idx: int32 [B][T][K]; o_g: fp32 [B][T][H][d_v];
 * lse_g: fp32 [B][T][H]. Limits: H % 16 == 0, H <= 64, d_v == 512, K <= 4096.
 * Indices outside [-1, n_stride) are skipped and set CSA2_DEV_BAD_INDEX.
 * Range of q: the products run on fp16 tensor cores, so q must be finite with
 * |q| <= 65504 (every such bf16 value is exact in fp16 down to 2^-14 in
 * magnitude; smaller ones round to fp16's subnormal grid, an absolute error of at
 * most 2^-25). A value outside sets CSA2_DEV_RANGE; the outputs of that query are
 * then undefined. The FP4 entries always fit (|C| <= 6 * 448).
 */
CSA2_API int csa2_sparse_decode(int B, int T, int H, const void* q,
                       const uint8_t* kv_codes, const uint8_t* kv_scales, int64_t n_stride,
                       const int32_t* idx, int K, int d_v, float softmax_scale,
                       float* o_g, float* lse_g, void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_swa_merge - sliding-window branch and its log-sum-exp merge.
 *
 * For each query, attends (same head/score convention as sparse_decode) over
 * the raw bf16 rows swa_kv[b, win_start[b*T+t] + r, :] for r < win_len[b*T+t]
 * (keys: 576 channels, values: first d_v), then combines with the global
 * branch as one softmax over the union of both key sets:
 *   LSE = logaddexp(LSE_g, LSE_s),  O = e^(LSE_g-LSE) O_g + e^(LSE_s-LSE) O_s.
 * swa_kv: bf16 [B][s_stride][576]; win_start, win_len: int32 [B*T] with
 * 0 <= win_len <= n_win <= 256; o_g, lse_g: the global branch (may be the
 * outputs of csa2_sparse_decode); o_out: fp32 [B][T][H][d_v] (may alias
 * o_g); lse_out: fp32 [B][T][H] (nullable, may alias lse_g).
 * A window outside [0, s_stride) is clipped and sets CSA2_DEV_BAD_WINDOW.
 * Range: q and the window rows must be finite with |x| <= 65504, as in
 * csa2_sparse_decode (fp16 tensor cores); a value outside sets CSA2_DEV_RANGE.
 */
CSA2_API int csa2_swa_merge(int B, int T, int H, const void* q,
                   const void* swa_kv, int64_t s_stride,
                   const int32_t* win_start, const int32_t* win_len, int n_win,
                   int d_v, float softmax_scale, const float* o_g, const float* lse_g,
                   float* o_out, float* lse_out, void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_decode_attention - both attention branches of a decode step in one call:
 * one softmax over the union of the selected FP4 entries (as csa2_sparse_decode)
 * and the window rows (as csa2_swa_merge), which equals csa2_sparse_decode
 * followed by csa2_swa_merge (the log-sum-exp merge of the two branches is the
 * softmax over both key sets; CSA2 sparse + sliding-window attention, blog repost).
 * Arguments as in those two calls; o: fp32 [B][T][H][d_v], lse: fp32 [B][T][H]
 * (nullable). Limits: H % 16 == 0, H <= 64, d_v == 512, K <= 4096, n_win <= 256.
 * An empty selection and an empty window give O = 0 and LSE = -inf. ws: the
 * 256-byte status header is enough; csa2_workspace_bytes(B, T, H, 0, K) bytes also
 * hold the split exchange (faster with few queries). q and the window rows: finite, |x| <= 65504
 * (CSA2_DEV_RANGE otherwise, as in csa2_sparse_decode).
 */
CSA2_API int csa2_decode_attention(int B, int T, int H, const void* q,
                   const uint8_t* kv_codes, const uint8_t* kv_scales, int64_t n_stride,
                   const int32_t* idx, int K, const void* swa_kv, int64_t s_stride,
                   const int32_t* win_start, const int32_t* win_len, int n_win, int d_v,
                   float softmax_scale, float* o, float* lse, void* ws, size_t ws_bytes,
                   void* stream);

/*
 * csa2_decode_layer - one CSA2 decode layer: csa2_index_topk followed by
 * csa2_decode_attention over the selection it writes (CSA2 global attention with
 * its indexer and top-K, picx.dev summary; the sliding-window branch, blog repost).
 *
 * Equals csa2_index_topk followed by csa2_decode_attention with the same
 * arguments (out_scores not written): out_idx [B][T][K] receives the selection
 * (REUSE: a copy of prev_idx), then o and lse the attention over it. kv_codes /
 * kv_scales and z share n_stride (one entry per compressed position).
 * Limits and argument rules: those of both calls. Both are checked before
 * anything is launched. ws: csa2_workspace_bytes(B, T, H, n_stride, K) bytes
 * prepared by csa2_workspace_init (REUSE: the header).
 */
CSA2_API int csa2_decode_layer(int mode, int B, int T, int H, int H_I, const void* q,
                   const void* q_idx, const float* w_idx, const void* z,
                   const uint8_t* kv_codes, const uint8_t* kv_scales, int64_t n_stride,
                   const int32_t* n_visible, int K, const int32_t* prev_idx, int32_t* out_idx,
                   const void* swa_kv, int64_t s_stride, const int32_t* win_start,
                   const int32_t* win_len, int n_win, int d_v, float softmax_scale, float* o,
                   float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_cache_append - decode-time cache append: one new token per sequence b
 * (the sliding window covers the most recent n_win tokens, blog repost; one
 * compressed entry per four tokens, wesearch.press card; FP4 entries, picx.dev
 * summary, Methodology / 5).
 *
 * The new token of sequence b has position p = n_tokens[b] (0-based; p < 0: the
 * sequence is idle and nothing is written for it). For each active b:
 *  - window: swa_row [B][576] bf16 is copied to rows p % n_win and
 *    p % n_win + n_win of swa_kv [B][s_stride][576] (a ring of n_win slots kept
 *    twice, s_stride >= 2 * n_win), so that after the call the last
 *    len = min(p + 1, n_win) tokens, oldest first, are the rows
 *    [win_start[b], win_start[b] + len) with win_start[b] = (p + 1 - len) % n_win
 *    and win_len[b] = len, the window arguments of csa2_swa_merge /
 *    csa2_decode_attention / csa2_decode_layer (T = 1);
 *  - entry: when (p + 1) % ratio == 0 the token completes entry
 *    e = (p + 1) / ratio - 1: entry_kv [B][576] (entry_dtype fp32 or bf16; how
 *    tokens become an entry is the caller's) is quantised as csa2_encode_kv (a)
 *    into kv_codes / kv_scales row [b][e] of [B][n_stride], and
 *    entry_z [B][64] bf16 is copied to z [B][n_stride][64] row e; an entry past
 *    the cache (e >= n_stride) is skipped and sets CSA2_DEV_BAD_INDEX;
 *  - n_visible[b] = (p + 1) / ratio (the entries visible to this token);
 *  - advance != 0: n_tokens[b] = p + 1 afterwards (call it with advance on the
 *    last of a step's per-layer appends).
 * Every output part is optional: swa_row == NULL skips the window rows,
 * entry_kv / entry_z == NULL skip those writes, n_visible / (win_start, win_len)
 * == NULL skip those outputs (win_start and win_len come together). ratio >= 1.
 * Alignment: 16 bytes for swa_row, swa_kv, entry_kv, entry_z, z; 8 for kv_codes.
 * ws: the 256-byte status header (csa2_workspace_init). The call waits for the
 * preceding kernel on the stream before writing (a ring row it replaces may
 * still be read by the previous step's attention).
 */
CSA2_API int csa2_cache_append(int B, int32_t* n_tokens, int advance, int ratio,
                   const void* swa_row, void* swa_kv, int64_t s_stride, int n_win,
                   const void* entry_kv, int entry_dtype, const void* entry_z,
                   uint8_t* kv_codes, uint8_t* kv_scales, void* z, int64_t n_stride,
                   int32_t* n_visible, int32_t* win_start, int32_t* win_len,
                   void* ws, size_t ws_bytes, void* stream);

/*
 * csa2_check_bounded_wait - self-check of the failure path of the kernels' waits.
 *
 * Every mbarrier wait inside the kernels gives up after one second of wall time,
 * sets CSA2_DEV_PIPELINE_TIMEOUT in the workspace status word, drains what it
 * started and returns (no kernel traps or spins). This call runs that path on
 * purpose: one CTA waits, through the same wait routine, on an mbarrier that
 * nothing arrives on, for limit_ns nanoseconds (1000 <= limit_ns <= 1e9), then sets
 * the bit and returns. Afterwards csa2_read_device_status reports CSA2_ERR_TIMEOUT
 * with that bit, and the context stays usable. ws: the 256-byte status header.
 */
CSA2_API int csa2_check_bounded_wait(int64_t limit_ns, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes that cover every call above with these or smaller sizes: a
 * 256-byte header (the device status word), then for csa2_index_topk two uint32
 * score-range words per query (B*T*8 bytes rounded up to 256), the fp32 indexer
 * scores ([B*T][n_max rounded up to 1024]) and the REINDEX_POOL block lists, and
 * last, when B*T <= 128, the attention calls' split exchange (512 KiB per query:
 * with few queries each query's keys are split over a cluster of 2 or 4 CTAs, whose
 * partial outputs meet in the last nsplit x 128 KiB per query of the workspace).
 * The attention calls need only the header: with less room than the exchange
 * (past the header and the range words) the splits merge through distributed
 * shared memory instead, which is slower. One workspace serves one stream at a
 * time. */
CSA2_API size_t csa2_workspace_bytes(int B, int T, int H, int64_t n_max, int K);

/* Zero the whole workspace (status word and score-range words) once after
 * allocation; the calls keep the range words at zero between calls. */
CSA2_API int csa2_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronise `stream`, copy the device status word to *flags (host pointer,
 * nullable) and clear it. Returns CSA2_OK when no bit was set,
 * CSA2_ERR_TIMEOUT when only CSA2_DEV_TOPK_LEVELS and/or
 * CSA2_DEV_PIPELINE_TIMEOUT are set, and CSA2_ERR_DEVICE_CHECK otherwise.
 */
CSA2_API int csa2_read_device_status(void* ws, void* stream, uint32_t* flags);

/* Static text for a csa2_status value. */
CSA2_API const char* csa2_status_string(int status);

/* Text of the last CUDA error a call on this thread turned into CSA2_ERR_CUDA
 * (static storage; "no error" before the first one). */
CSA2_API const char* csa2_last_cuda_error(void);

/* Library ABI version (major * 100 + minor). */
CSA2_API int csa2_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H_ */
