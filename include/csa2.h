/*
 * libcsa2 — C ABI of the CSA2 FP4 compressed global KV cache on B300 (sm_103a).
 *
 * The library implements the three data-parallel steps of the compressed global KV
 * cache of a CED/CSA2 decoder as described for DeepSeek-V4.1-Flash:
 *   - the write path: the CED projection C_l = H_{L/2} W_l^KV (tech-report digest,
 *     jiwasawa.github.io, section "Causal Encoder-Decoder (CED) アーキテクチャ",
 *     the equation there), quantised on write to FP4 E2M1 with one E4M3 scale per
 *     16 channels (ai2.x.ezic.info blog, section "KVを捨てる、共有する、作り直す");
 *   - the CSA2 indexer in Full, Reindex and Reuse modes with the hierarchical
 *     candidate pool (digest, section "Compressed Sparse Attention 2 (CSA2) による
 *     極限のKV cache圧縮"; zaikei.co.jp article, section "CSA2とFP4でキャッシュを圧縮");
 *   - the read path: gather + dequantise + sparse attention over the selected
 *     entries (zaikei article, same section: the cache is dequantised before
 *     attention; digest, "Reuse Mode").
 *
 * Conventions for every call:
 *   - All data pointers are DEVICE pointers unless a parameter says "host".
 *     bf16 values are passed as raw 16-bit patterns (uint16_t).
 *   - The caller owns every buffer.  Except where a function says otherwise, the
 *     library allocates no device memory; scratch is passed in as `workspace`,
 *     sized by the *_workspace_size queries.
 *   - Calls are asynchronous and ordered on `stream`.  The library keeps no state
 *     between calls and may be called from several host threads.
 *   - Host-detectable errors (null pointers, misalignment, unsupported sizes) return
 *     at once, before any launch.  Problems found on the device (an index outside
 *     its sequence, a page id outside the pool, a slot outside the pool, a wait
 *     that exceeded its limit) never abort a kernel: the offending entry is skipped
 *     and a CSA2_DEV_* bit is OR-ed into *dev_status (a device int32 the caller
 *     zeroes once and reads with csa2_read_status).  dev_status may be NULL, in
 *     which case such problems go unreported.
 *   - No call traps, asserts on the device, or throws across the ABI.
 *
 * Fixed geometry (checked, CSA2_ERR_UNSUPPORTED otherwise): latent width 512,
 * 16 channels per scale, indexer head dim 128 with 4 heads, 16 attention query
 * heads over the shared latent (MQA, head dim 512), 64 tokens per page.
 *
 * Layouts in HBM (one pool per Full-layer group; slot = page_id * 64 + token % 64):
 *   codes   uint8  [num_pages * 64][256]   E2M1 pairs, channel 2j in the low nibble
 *                                          of byte j, 2j+1 in the high nibble
 *   scales  uint8  [num_pages * 64][32]    E4M3 (OCP E4M3FN) bytes, one per 16 channels
 *   k_idx   bf16   [num_pages * 64][128]   indexer keys
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cudaStream_t; /* same opaque type as the CUDA runtime's */

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, misaligned buffer      */
  CSA2_ERR_UNSUPPORTED = 2,      /* a geometry this build does not implement        */
  CSA2_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed            */
  CSA2_ERR_DEVICE_FAULT = 4,     /* csa2_read_status: a CSA2_DEV_* fault bit was set */
  CSA2_ERR_TIMEOUT = 5           /* csa2_read_status: a bounded device wait expired */
} csa2_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define CSA2_DEV_BAD_INDEX 0x1 /* selected index outside [-1, seq_len) or pool entry out of range */
#define CSA2_DEV_BAD_PAGE 0x2  /* page-table entry outside [0, num_pages)                        */
#define CSA2_DEV_BAD_SLOT 0x4  /* write slot outside [0, num_slots)                              */
#define CSA2_DEV_TIMEOUT 0x8   /* a bounded wait (mbarrier) exceeded its iteration limit          */
#define CSA2_DEV_BAD_QSEQ 0x10 /* q_seq entry outside [0, num_seqs) or not non-decreasing         */

/* CSA2 layer modes (digest, section "CSA2": each layer is statically assigned one). */
typedef enum {
  CSA2_FULL = 0,    /* score every context token with this layer's indexer query; new top-K
                       and (optionally) the hierarchical candidate pool                    */
  CSA2_REINDEX = 1, /* re-score only the pool of the most recent Full layer, with that
                       layer's keys and this layer's query; new top-K                        */
  CSA2_REUSE = 2    /* inherit the indices of the most recent Full/Reindex layer            */
} csa2_mode;

/* Paged cache geometry.  All pointers are device pointers. */
typedef struct {
  int32_t num_seqs;          /* B                                                       */
  const int32_t* seq_lens;   /* [B] context tokens per sequence (>= 0)                   */
  const int32_t* page_table; /* [B][max_pages_per_seq] physical page id of logical page  */
  int32_t max_pages_per_seq; /* row length of page_table                                 */
  int32_t num_pages;         /* physical pages in each pool                              */
  int32_t page_size;         /* tokens per page; must be 64                              */
} csa2_pages;

/* Per-call indexer arguments. */
typedef struct {
  int32_t num_q;             /* query tokens in the batch                                */
  const int32_t* q_seq;      /* [num_q] sequence of each query, non-decreasing (device)  */
  int32_t max_q_per_seq;     /* host bound on queries per sequence, 1..4; > 1 selects the
                                tensor-core batched scoring of speculative draft tokens   */
  int32_t pool_size;         /* P: FULL writes top-min(P, N) into `pool` when pool != NULL;
                                REINDEX reads P entries per query from `pool`             */
  const int32_t* inherit_idx;/* REUSE: [num_q][topk] indices to inherit                   */
  void* workspace;           /* scratch, >= csa2_index_workspace_size() bytes, 256-B aligned */
  size_t workspace_bytes;
  int32_t* dev_status;       /* device int32 status word, may be NULL                    */
} csa2_index_args;

/* ------------------------------------------------------------------ write path ----
 * CED projection + quantise on write (digest, "Causal Encoder-Decoder (CED)": the
 * decoder's global KV is projected from the encoder's final hidden state,
 * C_l = H_{L/2} W_l^KV; blog: stored as FP4 E2M1 with an E4M3 scale per 16 channels).
 *
 *   H      bf16 [T][d_model]                 encoder final hidden state, row-major
 *   Wt     bf16 [n_out][d_model]              all projections stacked output-major
 *          (Wt[n][k] = W[k][n]); n_out = n_kv_proj*512 + n_idx_proj*128, first the
 *          n_kv_proj latent projections (512 columns each), then the n_idx_proj
 *          indexer-key projections (128 columns each)
 *   codes  uint8 [n_kv_proj][num_slots][256] output pools, one per latent projection
 *   scales uint8 [n_kv_proj][num_slots][32]
 *   k_idx  bf16  [n_idx_proj][num_slots][128] (may be NULL iff n_idx_proj == 0)
 *   slot_of_token int32 [T] physical row of each token, in [0, num_slots)
 *
 * Arithmetic: C = H.W with fp32 accumulation on the tensor cores; per token and
 * 16-channel block s = E4M3_RNE_satfinite(amax/6), codes = E2M1_RNE_sat(C/s) (IEEE
 * division, sign kept, s == 0 gives zero codes); indexer keys = bf16_RNE(C).
 * Any T >= 1 (the prefill of a whole prompt, or decode-time append of one new token per
 * sequence, each at its own slot); requires d_model % 64 == 0, 16-B aligned H and Wt.
 * Tokens whose slot is out of range are skipped (CSA2_DEV_BAD_SLOT).
 */
CSA2_API csa2_status csa2_kv_write(const uint16_t* H, const uint16_t* Wt, uint8_t* codes, uint8_t* scales,
                          uint16_t* k_idx, int32_t T, int32_t d_model, int32_t n_kv_proj,
                          int32_t n_idx_proj, const int32_t* slot_of_token, int64_t num_slots,
                          int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------ indexer -------
 * One CSA2 layer's index step (digest, section "CSA2" modes and "Hierarchical Sparse
 * Indexer").  Score of context token s for a query with indexer heads q_h (bf16
 * [4][128]): score_s = sum_{h<4} max(0, q_h . k_s), fp32 accumulation.  Positive
 * per-head weights are folded into q_h by the caller.  Ranking is (score descending,
 * token ascending).
 *
 *   FULL:    scores all N = seq_len tokens of the query's sequence; writes
 *            out_idx[q][0..K) = top-min(K, N) tokens, ascending, -1 padded, and, when
 *            pool != NULL and pool_size > 0, pool[q][0..P) = top-min(P, N) likewise.
 *   REINDEX: reads pool[q][0..P) (ascending, -1 padded, as a FULL call wrote it);
 *            scores only its valid entries with this layer's q_idx and the k_idx pool
 *            of the Full layer; out_idx = top-min(K, #valid) of the pool.
 *   REUSE:   out_idx = inherit_idx (one device copy; nothing if the pointers match).
 *
 *   q_idx   bf16 [num_q][4][128]     (unused by REUSE)
 *   k_idx   bf16 key pool [num_pages*64][128] of the Full layer (unused by REUSE)
 *   pool    int32 [num_q][pool_size]  FULL: output (nullable); REINDEX: input
 *   out_idx int32 [num_q][topk]
 * Workspace: csa2_index_workspace_size(mode, ...) bytes.
 */
CSA2_API csa2_status csa2_index(csa2_mode mode, const uint16_t* q_idx, const uint16_t* k_idx, int32_t* pool,
                       int32_t topk, int32_t* out_idx, const csa2_pages* pages,
                       const csa2_index_args* args, cudaStream_t stream);

CSA2_API size_t csa2_index_workspace_size(csa2_mode mode, int32_t num_q, int32_t max_pages_per_seq,
                                 int32_t pool_size);

/* ------------------------------------------------------------------ read path -----
 * Gather-dequantise sparse attention (zaikei article: the FP4 cache is dequantised
 * before attention; digest "Reuse Mode": sparse attention over the top-K entries).
 * MQA over the shared latent: K = V = c_hat_s = e2m1(code) * e4m3(scale) (exact).
 *   out[q][h] = sum_s softmax_s(softmax_scale * q_h . c_hat_s) c_hat_s
 *   lse[q][h] = natural-log sum-exp of the scaled logits
 * over the valid entries s of idx[q] (-1 entries are skipped).  A query with no valid
 * entry gets out = 0 and lse = -inf.
 *
 *   q      bf16 [num_q][16][512]
 *   codes, scales  the Full layer's pools (layout above)
 *   idx    int32 [num_q][topk], entries in [-1, seq_len); 1 <= topk <= CSA2_ATTN_MAX_TOPK
 *          (CSA2_ERR_UNSUPPORTED above it)
 *   out    fp32 [num_q][16][512];  lse fp32 [num_q][16] (nullable)
 *   q_seq  int32 [num_q]
 * Workspace: csa2_attn_workspace_size(num_q, topk) bytes (may be 0).
 * Arithmetic: the logits are taken on the block-scaled FP4 tensor cores from the codes
 * and scales as stored, against q written as six NVFP4 terms (|q - terms| <= (3/16)^6 of
 * each 16-channel block's maximum), with fp32 accumulation; fp32 online softmax (exp2),
 * split over the selected set and merged by log-sum-exp; the weighted sum uses the
 * softmax weights as f16 high + low parts against the exactly dequantised rows, with
 * fp32 accumulation.  Outputs agree with the exact definition within 2e-3 x RMS(out).
 */
#define CSA2_ATTN_MAX_TOPK 65536
CSA2_API csa2_status csa2_sparse_attn(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                             const int32_t* idx, const csa2_pages* pages, float* out, float* lse,
                             int32_t num_q, const int32_t* q_seq, int32_t topk, float softmax_scale,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status,
                             cudaStream_t stream);

CSA2_API size_t csa2_attn_workspace_size(int32_t num_q, int32_t topk);

/* csa2_sparse_attn over an MXFP4 cache (tech-report digest, "FP4 メイン KV Cache と SWA
 * Bounded Replay": OCP MXFP4, E2M1 elements; read as one E8M0 scale per 32 channels, the
 * layout csa2_quantize_mx writes): scales uint8 [num_pages*64][16], c_hat = e2m1(code) *
 * 2^(byte - 127).  Same arguments, workspace and results otherwise.  The kernel rebases
 * every split's scales on their largest byte `ref`; a value is represented exactly when
 * its scale byte is at least ref - 23, and contributions more than 2^23 below the
 * split's largest scale lose precision or vanish. */
CSA2_API csa2_status csa2_sparse_attn_mx(const uint16_t* q, const uint8_t* codes,
                                         const uint8_t* scales, const int32_t* idx,
                                         const csa2_pages* pages, float* out, float* lse,
                                         int32_t num_q, const int32_t* q_seq, int32_t topk,
                                         float softmax_scale, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_status,
                                         cudaStream_t stream);

/* Multi-query sparse attention, dense-contraction form: the queries come in chunks of
 * `chunk` consecutive queries (1..4) of one sequence -- the draft tokens of a decode step,
 * or consecutive positions of a prefill chunk -- each with its own top-K selection
 * (tech-report digest, "Reuse Mode": attention over each query's top-K entries;
 * "Hierarchical Sparse Indexer": the search and its cost are per query; draft tokens:
 * the digest's DSpark item under "さらなるアーキテクチャ拡張技術", speculative decoding
 * with semi-autoregressive drafts; prefill: the zaikei article's 64K-token sparse
 * attention training length).
 * The union of a chunk's selections is gathered and dequantised once, and all the
 * chunk's heads are contracted against it on the tensor cores, each query's logits
 * masked to the entries it selected.  Results equal csa2_sparse_attn on the same
 * arguments (same formula, rounding order aside), for selections without a repeated
 * token: a token listed twice by one query counts once here.
 *
 *   chunk  1..4; num_q a multiple of chunk; every query of a chunk has the same q_seq
 *          (otherwise CSA2_DEV_BAD_QSEQ and that chunk's queries get out = 0, lse = -inf)
 *   topk   chunk * topk <= CSA2_CHUNK_ATTN_MAX_UNION (CSA2_ERR_UNSUPPORTED above it)
 *   other arguments as csa2_sparse_attn (E4M3 / 16 cache); lse nullable
 * Workspace: csa2_chunk_attn_workspace_size(num_q, chunk, topk) bytes (16-byte aligned).
 */
#define CSA2_CHUNK_ATTN_MAX_UNION 8192
CSA2_API csa2_status csa2_sparse_attn_chunked(const uint16_t* q, const uint8_t* codes,
                                              const uint8_t* scales, const int32_t* idx,
                                              const csa2_pages* pages, float* out, float* lse,
                                              int32_t num_q, const int32_t* q_seq, int32_t chunk,
                                              int32_t topk, float softmax_scale, void* workspace,
                                              size_t workspace_bytes, int32_t* dev_status,
                                              cudaStream_t stream);

/* Workspace bytes of csa2_sparse_attn_chunked; 0 for arguments it rejects. */
CSA2_API size_t csa2_chunk_attn_workspace_size(int32_t num_q, int32_t chunk, int32_t topk);

/* csa2_sparse_attn without caller workspace.  The pages have no counterpart to this
 * entry point: it exists for callers that cannot allocate device memory around the
 * call (plain C clients that hold no device allocator, or decode loops that must not
 * call cudaMalloc / cudaFree, which can synchronise the device, while work is in flight).
 *
 * Same arguments, arithmetic and results as csa2_sparse_attn.  The split partials go
 * to a fixed device array of CSA2_ATTN_STATIC_SCRATCH_BYTES inside this library; the
 * call allocates nothing.  The first call on a device, made with that device current,
 * resolves the array's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture.  Returns CSA2_ERR_UNSUPPORTED when
 * csa2_attn_workspace_size(num_q, topk) exceeds CSA2_ATTN_STATIC_SCRATCH_BYTES -- on a
 * 148-SM B300 that is more than 74 queries at topk 2048 (64 queries need 9.8 MiB) -- and
 * CSA2_ERR_CUDA if the address cannot be resolved.  The array is shared by all calls
 * on a device: calls that overlap in time (several streams or host threads) race; calls
 * issued one after another on one stream do not, so a batch over the limit can be split
 * into several calls on one stream.  The address is resolved again after the device's
 * context is destroyed and recreated (cudaDeviceReset).  Footprint: the array occupies
 * CSA2_ATTN_STATIC_SCRATCH_BYTES of device memory on every device where it is loaded --
 * at the first call of this function on the device under lazy module loading (the CUDA
 * default), or at context creation under CUDA_MODULE_LOADING=EAGER even if the function
 * is never called -- and until the context is destroyed. */
#define CSA2_ATTN_STATIC_SCRATCH_BYTES (16u << 20)
CSA2_API csa2_status csa2_sparse_attn_static(const uint16_t* q, const uint8_t* codes,
                                             const uint8_t* scales, const int32_t* idx,
                                             const csa2_pages* pages, float* out, float* lse,
                                             int32_t num_q, const int32_t* q_seq, int32_t topk,
                                             float softmax_scale, int32_t* dev_status,
                                             cudaStream_t stream);

/* ------------------------------------------------------------------ codec ---------
 * Standalone quantise / dequantise of latent rows (blog: E2M1 values, one E4M3 scale
 * per 16 channels).  Same arithmetic as the write path's epilogue.
 *   x      fp32 [T][D], D % 16 == 0, D <= 4096, 16-B aligned
 *   slot_of_token int32 [T] destination / source row in [0, num_slots)
 *   codes  uint8 [num_slots][D/2];  scales uint8 [num_slots][D/16]
 */
CSA2_API csa2_status csa2_quantize(const float* x, const int32_t* slot_of_token, uint8_t* codes,
                          uint8_t* scales, int32_t T, int32_t D, int64_t num_slots,
                          int32_t* dev_status, cudaStream_t stream);
CSA2_API csa2_status csa2_dequantize(const uint8_t* codes, const uint8_t* scales,
                            const int32_t* slot_of_token, float* x, int32_t T, int32_t D,
                            int64_t num_slots, int32_t* dev_status, cudaStream_t stream);

/* MXFP4 variant of the codec (tech-report digest, "FP4 メイン KV Cache と SWA Bounded
 * Replay": the main KV in the OCP-standard MXFP4 format, E2M1 elements), read as OCP MX:
 * one E8M0 scale byte per 32 channels, X = 2^(floor(log2 amax) - 2) clamped to
 * 2^-127 .. 2^127 (byte = exponent + 127); codes = E2M1_RNE_satfinite(x / X), sign kept;
 * a block whose amax is 0 gets scale byte 0 and zero codes.  Dequantised values are
 * e2m1(code) * 2^(byte - 127) in fp32 (exact within fp32's range).  272 B per 512
 * channels against 288 B for E4M3 / 16.
 *   x      fp32 [T][D], D % 32 == 0, D <= 4096, 16-B aligned
 *   slot_of_token int32 [T] destination / source row in [0, num_slots)
 *   codes  uint8 [num_slots][D/2], 16-B aligned;  scales uint8 [num_slots][D/32]
 */
CSA2_API csa2_status csa2_quantize_mx(const float* x, const int32_t* slot_of_token, uint8_t* codes,
                                      uint8_t* scales, int32_t T, int32_t D, int64_t num_slots,
                                      int32_t* dev_status, cudaStream_t stream);
CSA2_API csa2_status csa2_dequantize_mx(const uint8_t* codes, const uint8_t* scales,
                                        const int32_t* slot_of_token, float* x, int32_t T,
                                        int32_t D, int64_t num_slots, int32_t* dev_status,
                                        cudaStream_t stream);

/* ------------------------------------------------------------------ persistent tier -
 * Export / import of whole cache pages for the persistent KV tier (zaikei article,
 * opening section: the persistent KV cache that resumes sessions lives on SSD or in host
 * memory; tech-report digest, "FP4 メイン KV Cache と SWA Bounded Replay": the
 * sliding-window KV is left out of it, so what persists is the global cache).  A page
 * record holds the page's 64 tokens:
 *   codes [64][256] u8 | scales [64][S] u8 | keys [64][128] bf16
 * with S = scale_row_bytes: 32 for E4M3 per 16 channels, 16 for the MXFP4 variant.
 * Records are packed back to back in page_ids order; csa2_page_export_bytes(S) is the
 * record size (34816 or 33792 B), 0 for any other S.
 *   codes, scales, keys  the pools of one Full group ([num_pages*64][256], [..][S],
 *          [..][128] bf16), 16-B aligned
 *   page_ids int32 [n_pages] (device) physical pages to export from / import into
 *   packed  n_pages records, 16-B aligned, device memory or host memory the GPU can
 *          address (mapped pinned memory)
 * Export copies the pages into `packed`; import copies the records into the pages.  Page
 * ids outside [0, num_pages) set CSA2_DEV_BAD_PAGE: export writes a zero record, import
 * skips it.  S other than 16 or 32 returns CSA2_ERR_UNSUPPORTED. */
CSA2_API size_t csa2_page_export_bytes(int32_t scale_row_bytes);
CSA2_API csa2_status csa2_export_pages(const uint8_t* codes, const uint8_t* scales,
                                       const uint16_t* keys, int32_t scale_row_bytes,
                                       int64_t num_pages, const int32_t* page_ids, int32_t n_pages,
                                       uint8_t* packed, int32_t* dev_status, cudaStream_t stream);
CSA2_API csa2_status csa2_import_pages(const uint8_t* packed, int32_t scale_row_bytes,
                                       const int32_t* page_ids, int32_t n_pages, int64_t num_pages,
                                       uint8_t* codes, uint8_t* scales, uint16_t* keys,
                                       int32_t* dev_status, cudaStream_t stream);

/* ------------------------------------------------------------------ status --------
 * Synchronises `stream`, copies *dev_status to *host_bits (host, nullable), resets
 * the device word to 0 and returns CSA2_ERR_TIMEOUT if CSA2_DEV_TIMEOUT was set,
 * CSA2_ERR_DEVICE_FAULT if any other bit was set, CSA2_OK otherwise. */
CSA2_API csa2_status csa2_read_status(int32_t* dev_status, int32_t* host_bits, cudaStream_t stream);

/* ------------------------------------------------------------------ diagnostic ----
 * Exercises the failure-detection contract on the device without a fault.  One warp
 * waits, with the bounded mbarrier wait every TMA- or tcgen05-fed kernel of this library
 * uses, on a barrier phase that completes only if `arrive` is nonzero.  With arrive = 0
 * the wait gives up after `limit` polls (1 <= limit <= 2^20; each poll may suspend for a
 * hardware-chosen interval, so 2^20 polls stay well under a second), ORs CSA2_DEV_TIMEOUT
 * into *dev_status and the kernel returns; nothing is left in flight and the context
 * stays usable.  With arrive != 0 the wait completes and nothing is reported.
 * Returns CSA2_ERR_INVALID_ARGUMENT for a null dev_status or a limit out of range. */
CSA2_API csa2_status csa2_check_bounded_wait(int32_t arrive, uint32_t limit, int32_t* dev_status,
                                             cudaStream_t stream);

CSA2_API const char* csa2_status_string(csa2_status s);
CSA2_API int32_t csa2_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
