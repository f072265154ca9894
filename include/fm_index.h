/*
 * fm_index.h -- C ABI of the GB300 (sm_103a) Lookahead-Sparse-Attention c4
 * indexer library (libfm_index.so).
 *
 * The library computes the data-parallel hot path of the LSA indexer that
 * scores DeepSeek-V4 compressed c4 chunk keys:
 *   - the Memory Indexer score I = sigmoid(sum_h w_h * ReLU(q_h . K_s)), its
 *     OR-union over indexer layers and the resident-set bitmask;
 *   - the native lightning-indexer score sum_h w_h * ReLU(q_h . k_s) over the
 *     resident 64-chunk pages, followed by the top-k (k <= 1024, normally 512);
 *   - the same score for many prefill queries against dense chunk keys under
 *     the causal chunk limit, followed by the top-k;
 *   - the top-k select itself over caller-provided scores.
 *
 * Sources (page titles as published):
 *   [FM] "FlashMemory-DeepSeek-V4: Lightning Index Ultra-Long Context via
 *        Lookahead Sparse Attention" (paper summary), sec. 3 "Memory Indexer
 *        scoring function" (I_{t,s}, the 0.5 threshold, the union over layers
 *        10/12/20, R_t[s] = 1(max_l I^(l) >= 0.5)), sec. 6 (Mode A/B, Level 2
 *        top-512 inside the resident set).
 *   [RM] "FlashMemory-DeepSeek-V4" (repository README): "Retriever
 *        architecture" (score formula, fused_w), "compressed_k format" (E4M3
 *        key bytes + fp32 per-chunk scale, dequant = fp8.float() * scale),
 *        "Two-level recall algorithm" (Level 1 / Level 2), key-optimisations
 *        table ("Two-level recall", "Page-recall": 64-chunk pages).
 *   [V4] "DeepSeek-V4 CSA + HCA explained": sec. 3 "C4Indexer" (n_heads = 64,
 *        head_dim = 128, index_topk = 512; CSA-1 score, CSA-2 top-512), sec. 8
 *        (4 tokens per c4 chunk; fewer than 512 chunks -> take them all).
 *
 * Conventions for every entry point
 *   - Array pointers are caller-owned DEVICE memory unless stated otherwise;
 *     the library never frees or retains them.  Layouts are dense row-major in
 *     the order of the bracketed shape, except where a stride is passed.
 *   - bf16 tensors are passed as uint16_t bit patterns; E4M3 keys as uint8_t
 *     codes (OCP FP8 E4M3: bias 7, max 448, S.1111.111 = NaN).  Key codes must
 *     be finite: a chunk whose key holds the NaN code gets an unspecified
 *     logit (quantised keys never hold it).
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  The
 *     host validates every argument before the first launch; on a non-OK
 *     return nothing was enqueued (FM_ERR_CUDA: a launch failed; earlier
 *     launches of the same call may have been enqueued).
 *   - n_h must be 64 and d must be 128 (the C4Indexer's sizes).
 *   - Ties in a top-k are broken by the lower chunk id.  Selected ids are
 *     written in ascending id order and padded with -1 (scores with -inf).
 *   - Kernels never trap and never spin without a bound.  A device-detected
 *     problem (an out-of-range page id, a bounded wait that ran out) sets a
 *     bit in the library's device status word and the affected work is
 *     skipped; read it with fm_device_status() or, as a status code,
 *     fm_check_device_status().
 *   - Thread-safety: calls may be issued from several host threads; the last
 *     error message is thread-local.
 */
#ifndef FM_INDEX_H
#define FM_INDEX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fm_stream_t; /* == cudaStream_t */

typedef enum {
  FM_OK = 0,
  FM_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad size, unsupported n_h/d/k    */
  FM_ERR_UNSUPPORTED = 2,    /* current device is not an sm_103 GPU                        */
  FM_ERR_CUDA = 3,           /* a CUDA runtime/driver call failed (see fm_last_error)      */
  FM_ERR_DEVICE_BOUNDS = 4,  /* a kernel met an out-of-range or repeated page id and      */
                             /* skipped it (fm_check_device_status; FM_DEVERR_PAGE_RANGE,  */
                             /* FM_DEVERR_DUP_PAGE)                                        */
  FM_ERR_WORKSPACE = 5,      /* workspace pointer null/misaligned or smaller than needed   */
  FM_ERR_DEVICE_TIMEOUT = 6  /* a kernel's bounded on-chip wait ran out and the launch     */
                             /* gave up (fm_check_device_status; FM_DEVERR_TIMEOUT)        */
} fm_status;

/* Key element types of a paged key pool (fm_native_topk_paged's key_dtype). */
typedef enum {
  FM_DTYPE_BF16 = 1,     /* bf16 keys, no scale                                        */
  FM_DTYPE_FP8_E4M3 = 2  /* E4M3 codes with one fp32 dequant scale per chunk           */
} fm_dtype;

/* Bits of the device status word (fm_device_status). */
#define FM_PAGED_MAX_R 4096       /* page-table entries per query of the paged calls     */
#define FM_DEVERR_PAGE_RANGE 0x1u  /* page_phys outside [0, P): that page was skipped     */
#define FM_DEVERR_TIMEOUT 0x2u     /* a bounded on-chip wait ran out: the launch gave up  */
#define FM_DEVERR_DUP_PAGE 0x4u    /* repeated logical page in one query's page table     */

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
int fm_version(void);

/* Human-readable message for the last non-OK status returned on this thread. */
const char* fm_last_error(void);

/*
 * Memory Indexer score, OR-union over layers and resident bitmask
 * ([FM] sec. 3; [RM] "Retriever architecture", "Two-level recall", Level 1).
 *
 * For request b, layer l and chunk s:
 *     x[b,l,s] = sum_{h<n_h} w[b,l,h] * ReLU( sum_{j<d} q[b,l,h,j] * K[b,l,s,j] )
 * and the chunk is resident iff max_l sigmoid(x[b,l,s]) >= threshold, i.e. the
 * OR of the per-layer sets { s | sigmoid(x[b,l,s]) >= threshold }.
 *
 *   q           [B, L, n_h, d] bf16             per-layer query heads
 *   w           [B, L, n_h] fp32                fused head weights (the caller
 *                                               has applied any head_dim^-1/2 *
 *                                               n_h^-1/2 factor: [RM] fused_w)
 *   keys        bf16, element (b,l,s,j) at keys[b*key_stride_b + l*key_stride_l
 *               + s*d + j]; 16-byte aligned; strides multiples of 8 elements
 *   B >= 0, 1 <= L <= 4, S >= 0 (S < 2^31), n_h = 64, d = 128
 *   threshold   in (0, 1); 0.5 in the pages.  The device tests
 *               max_l x >= log(threshold / (1 - threshold)).
 *   mask_out    [B, ceil(S/32)] uint32: bit (s & 31) of word s >> 5 is chunk s;
 *               bits at s >= S are written as zero.   (required)
 *   maxsig_out  [B, S] fp32 max_l sigmoid(x), or NULL
 *   logits_out  [B, L, S] fp32 x, or NULL
 * Errors: FM_ERR_INVALID_ARG for any violated condition above.
 */
fm_status fm_memindex_score_mask(const uint16_t* q, const float* w, const uint16_t* keys,
                                 int64_t key_stride_b, int64_t key_stride_l, int B, int L, int64_t S,
                                 int n_h, int d, float threshold, uint32_t* mask_out, float* maxsig_out,
                                 float* logits_out, fm_stream_t stream);

/*
 * The same Memory Indexer over compressed keys ([FM] sec. 6 and [RM]
 * "compressed_k format": the retriever reads each chunk as 128 E4M3 bytes plus
 * an fp32 scale, dequantised as fp8.float() * scale):
 *     x[b,l,s] = sum_h w[b,l,h] * ReLU( q[b,l,h,:] . (scale[b,l,s] * e4m3(k8[b,l,s,:])) )
 * with the union, threshold and outputs of fm_memindex_score_mask.  The scale
 * is applied to each head's dot (equal up to one fp32 rounding per element).
 *
 *   k8          E4M3 codes, element (b,l,s,j) at k8[b*key_stride_b +
 *               l*key_stride_l + s*128 + j] (byte strides, multiples of 16;
 *               16-byte aligned)
 *   k_scale     fp32, (b,l,s) at k_scale[b*scale_stride_b + l*scale_stride_l + s]
 *   workspace   >= fm_memindex_fp8_workspace(B, L) bytes, 256-byte aligned
 *               (the split query and its weights: 20.3 KB per (request, layer))
 * Other arguments, outputs and errors as fm_memindex_score_mask;
 * FM_ERR_WORKSPACE for a missing or short workspace.
 */
size_t fm_memindex_fp8_workspace(int B, int L);
fm_status fm_memindex_score_mask_fp8(const uint16_t* q, const float* w, const uint8_t* k8, const float* k_scale,
                                     int64_t key_stride_b, int64_t key_stride_l, int64_t scale_stride_b,
                                     int64_t scale_stride_l, int B, int L, int64_t S, int n_h, int d,
                                     float threshold, uint32_t* mask_out, float* maxsig_out, float* logits_out,
                                     void* workspace, size_t workspace_bytes, fm_stream_t stream);

/*
 * The trained retriever's Memory Indexer ([RM] "Retriever architecture",
 * "compressed_k format", "Joint checkpoint + ensemble"): the logits of
 * fm_memindex_score_mask_fp8 with n_h = 128 (the retriever) or 64 heads, read
 * from packed compressed_k rows, and the per-layer sigmoid scores ensembled
 * per chunk by max (the union) or mean:
 *     e[b,s] = max_l sigmoid(x[b,l,s])  or  (1/L) sum_l sigmoid(x[b,l,s])
 *     resident[b,s] = e[b,s] >= threshold
 *
 *   q             [B, L, n_h, 128] bf16; w [B, L, n_h] fp32 (fused weights)
 *   compressed_k  chunk (b,l,s) is the 132 bytes at compressed_k +
 *                 b*ck_stride_b + l*ck_stride_l + s*132: 128 E4M3 key bytes,
 *                 then the fp32 scale (little-endian).  Byte strides are
 *                 multiples of 16 (so S % 4 == 0); 16-byte aligned.
 *   ensemble      FM_ENSEMBLE_MAX or FM_ENSEMBLE_MEAN
 *   threshold     in (0, 1)
 *   mask_out      as fm_memindex_score_mask (required)
 *   ens_out       [B, S] fp32 e[b,s], or NULL
 *   logits_out    [B, L, S] fp32 x, or NULL
 *   workspace     >= fm_retriever_workspace(B, L, n_h) bytes, 256-byte aligned
 *                 (the split query and weights: 36.5 KB per (request, layer)
 *                 at 128 heads)
 * Errors: FM_ERR_INVALID_ARG for n_h not 64/128, d != 128, L outside 1..4,
 * S % 4 != 0, a bad ensemble, threshold, pointer or stride; FM_ERR_WORKSPACE
 * for a missing or short workspace.
 */
#define FM_ENSEMBLE_MAX 0
#define FM_ENSEMBLE_MEAN 1
size_t fm_retriever_workspace(int B, int L, int n_h);
fm_status fm_retriever_score_mask(const uint16_t* q, const float* w, const uint8_t* compressed_k,
                                  int64_t ck_stride_b, int64_t ck_stride_l, int B, int L, int64_t S, int n_h,
                                  int d, int ensemble, float threshold, uint32_t* mask_out, float* ens_out,
                                  float* logits_out, void* workspace, size_t workspace_bytes, fm_stream_t stream);

/*
 * The query side of a CSA layer's indexer ([RM] "Retriever architecture",
 * "Hyperparameters"): from T tokens' hidden states to the query heads and head
 * weights the Memory Indexer / retriever score with.  For token t:
 *     a = wq_a . h_t                  Linear dim -> r, no bias
 *     c = RMSNorm(a; q_norm, eps)     c = a / sqrt(mean(a^2) + eps) * q_norm
 *     u = wq_b . c                    Linear r -> n_h * 128, reshaped [n_h, 128]
 *     q_h = H(RoPE(u_h, pos_t))       rotary (YaRN) on entries 64..127, pairs
 *                                     (64+2i, 65+2i), angle pos_t * theta'_i,
 *                                     then the normalised Walsh-Hadamard
 *                                     transform H (Sylvester order, / sqrt(128))
 *     w = (w_proj . h_t) / sqrt(128 * n_h)
 * theta'_i is YaRN's NTK-by-parts frequency of base^(-2i/64) (rope_base,
 * rope_factor, rope_orig_len, rope_beta_fast, rope_beta_slow; the retriever
 * uses 160000, 16, 65536, 32, 1).  The GEMMs take bf16 inputs with fp32
 * accumulation; the RMSNorm output is rounded to bf16 (wq_b's input type).
 *
 *   hidden   [T, dim] bf16;  wq_a [r, dim], q_norm [r], wq_b [n_h*128, r],
 *            w_proj [n_h, dim] bf16 (row-major [out, in]; 16-byte aligned)
 *   pos      [T] int64 token positions
 *   dim, r   multiples of 8; head_dim == 128; rope_dim == 64
 *   q_out    [T, n_h, 128] bf16 (required); q_out_f32 [T, n_h, 128] or NULL
 *   w_out    [T, n_h] fp32 (required)
 *   workspace >= fm_query_chain_workspace(T, r, n_h) bytes, 256-byte aligned
 * The projections run on the tensor cores with the weights streamed once
 * per 256 tokens; their K-split partial sums (in the workspace) are reduced
 * in a fixed order, so results do not depend on scheduling.
 * Errors: FM_ERR_INVALID_ARG for bad sizes, parameters or pointers;
 * FM_ERR_WORKSPACE; FM_ERR_CUDA for a launch failure.
 */
size_t fm_query_chain_workspace(int T, int r, int n_h);

/*
 * The query chain of L indexer layers (1 <= L <= 4) in one call: the layers'
 * projections share launches, so the fixed cost of a launch is paid once per
 * call rather than once per layer (the retriever scores its three indexer
 * layers together, [RM] "Retriever architecture").  Layer l computes
 * fm_query_chain from hidden[l] with its own weights wq_a[l], q_norm[l],
 * wq_b[l] and w_proj[l]; the T tokens and their positions are shared.
 *
 *   hidden, wq_a, q_norm, wq_b, w_proj   HOST arrays of L device pointers,
 *            each as in fm_query_chain
 *   q_out    [T, L, n_h, 128] bf16 (required) -- the layout
 *            fm_retriever_score_mask takes as q with B = T;
 *            q_out_f32 the same in fp32, or NULL
 *   w_out    [T, L, n_h] fp32 (required)
 *   workspace >= fm_query_chain_layers_workspace(L, T, r, n_h) bytes,
 *            256-byte aligned
 * fm_query_chain is this call with L = 1.  Errors as fm_query_chain, and
 * FM_ERR_INVALID_ARG for L outside 1..4.
 */
size_t fm_query_chain_layers_workspace(int L, int T, int r, int n_h);
fm_status fm_query_chain_layers(int L, const uint16_t* const* hidden, const uint16_t* const* wq_a,
                                const uint16_t* const* q_norm, const uint16_t* const* wq_b,
                                const uint16_t* const* w_proj, const int64_t* pos, int T, int dim, int r, int n_h,
                                int head_dim, int rope_dim, double rope_base, double rope_factor,
                                double rope_orig_len, double rope_beta_fast, double rope_beta_slow, float eps,
                                uint16_t* q_out, float* q_out_f32, float* w_out, void* workspace,
                                size_t workspace_bytes, fm_stream_t stream);
fm_status fm_query_chain(const uint16_t* hidden, const uint16_t* wq_a, const uint16_t* q_norm, const uint16_t* wq_b,
                         const uint16_t* w_proj, const int64_t* pos, int T, int dim, int r, int n_h, int head_dim,
                         int rope_dim, double rope_base, double rope_factor, double rope_orig_len,
                         double rope_beta_fast, double rope_beta_slow, float eps, uint16_t* q_out, float* q_out_f32,
                         float* w_out, void* workspace, size_t workspace_bytes, fm_stream_t stream);

/*
 * Top-k select over caller-provided scores ([FM] sec. 3 "Top-k" of the native
 * score; [V4] sec. 3 CSA-2 top-512).
 *
 *   scores      [rows, ld] fp32; row r has candidates 0 .. n_valid[r]-1
 *               (n_valid == NULL: every row has n candidates), n <= ld
 *   idx_out     [rows, k] int32: the min(k, n_r) best candidate indices by
 *               (score desc, index asc), ascending, padded with -1
 *   score_out   [rows, k] fp32 matching scores (-inf padding), or NULL
 *   1 <= k <= 1024; n < 2^31.  NaN scores rank as -inf; -0 equals +0.
 *   workspace   device scratch of at least fm_topk_workspace(rows, n) bytes,
 *               256-byte aligned (may be NULL when that size is 0; it is 0
 *               for every size in this version)
 */
size_t fm_topk_workspace(int rows, int64_t n);
fm_status fm_topk_select(const float* scores, int64_t ld, const int32_t* n_valid, int rows, int64_t n,
                         int k, int32_t* idx_out, float* score_out, void* workspace, size_t workspace_bytes,
                         fm_stream_t stream);

/*
 * Page recall: the densest resident pages of each request ([RM] "Two-level
 * recall algorithm", Level 1: resident_set = threshold + recent + sink;
 * "Page-recall": 64-chunk pages; the KMAX note under "Reference performance":
 * KMAX = 96 / 192 / 384 densest pages at 256K / 512K / 1M).
 *
 * For request b, chunk s < S is resident iff bit s & 31 of mask[b, s >> 5] is
 * set, or s < sink, or s >= S - recent.  Page p holds chunks 64p .. 64p + 63;
 * its density is its number of resident chunks.  The kmax pages of highest
 * density are recalled (pages of density 0 never are; equal densities go to
 * the lower page id).  This turns fm_memindex_score_mask's bitmask into the
 * page table that fm_native_topk_paged reads (logical page ids).
 *
 *   mask        [B, ceil(S/32)] uint32 (bits at s >= S are ignored)
 *   B >= 0, 0 <= S < 2^31, sink >= 0, recent >= 0 (each clamped to S),
 *   1 <= kmax <= 65536
 *   pages_out   [B, kmax] int32 recalled page ids, ascending, padded with -1
 *   density_out [B, kmax] int32 their densities (-1 padding), or NULL
 *   n_out       [B] int32 number of pages recalled, or NULL
 * Errors: FM_ERR_INVALID_ARG for any violated condition above.
 */
fm_status fm_page_recall(const uint32_t* mask, int B, int64_t S, int64_t sink, int64_t recent, int kmax,
                         int32_t* pages_out, int32_t* density_out, int32_t* n_out, fm_stream_t stream);

/*
 * Native lightning-indexer score over the resident pages + top-k
 * ([FM] sec. 3 C^CoreComp and sec. 6 Level 2; [RM] "Two-level recall" Level 2,
 * "Page-recall" 64-chunk pages, "compressed_k format"; [V4] sec. 3 CSA-1/2).
 *
 * Query qi scores the chunks of its first n_res[qi] page-table entries:
 *     y = sum_h w[qi,h] * ReLU( scale[p,o] * sum_j q[qi,h,j] * e4m3(k_pool[p,o,j]) )   (E4M3 pool)
 *     y = sum_h w[qi,h] * ReLU( sum_j q[qi,h,j] * k_pool[p,o,j] )                      (bf16 pool)
 * for pool page p = page_phys[qi,r] and offset o < 64; the chunk's id is
 * page_logical[qi,r] * 64 + o.  Chunks outside the listed pages are not
 * candidates (equivalent to Mode A's -inf).  The result does not depend on the
 * order of a query's page-table entries.
 *
 *   q            [Q, n_h, d] bf16, 16-byte aligned;  w [Q, n_h] fp32 (fused weights)
 *   k_pool       [P, 64, d], 16-byte aligned: E4M3 codes (key_dtype
 *                FM_DTYPE_FP8_E4M3, the compressed_k keys) or bf16 keys
 *                (FM_DTYPE_BF16)
 *   key_dtype    FM_DTYPE_FP8_E4M3 or FM_DTYPE_BF16
 *   k_scale      [P, 64] fp32 per-chunk dequant scale (E4M3); NULL for bf16
 *   page_phys    [Q, R] int32 pool page; entries outside [0, P) are skipped and
 *                flagged FM_DEVERR_PAGE_RANGE
 *   page_logical [Q, R] int32 logical page id in [0, 2^25); distinct within
 *                a query (a repeat is flagged FM_DEVERR_DUP_PAGE and skipped:
 *                the entry listed first is kept)
 *   n_res        [Q] int32 entries used per query (clamped to [0, R]), or NULL = R
 *   1 <= R <= FM_PAGED_MAX_R (4096 pages = 262144 chunks: the whole history
 *   of a 1M-token request, so the call also serves the full-history native
 *   top-k that scores every chunk), 1 <= k <= 1024, Q >= 0
 *   idx_out      [Q, k] int32 chunk ids; score_out [Q, k] fp32 or NULL
 *   workspace    >= fm_native_topk_paged_workspace(Q, R) bytes, 256-byte aligned
 */
size_t fm_native_topk_paged_workspace(int Q, int R);
fm_status fm_native_topk_paged(const uint16_t* q, const float* w, const void* k_pool, int key_dtype,
                               const float* k_scale, int64_t P, const int32_t* page_phys,
                               const int32_t* page_logical, const int32_t* n_res, int Q, int R, int n_h, int d,
                               int k, int32_t* idx_out, float* score_out, void* workspace, size_t workspace_bytes,
                               fm_stream_t stream);

/*
 * fm_native_topk_paged with the Level-2 resident mask and the fused remap
 * ([RM] "Two-level recall algorithm" Level 2: the native top-512 is confined
 * to the resident set by masking non-resident chunk logits to -inf; [FM]
 * sec. 6 Mode A; [RM] "Fused remap": top-512 columns map directly to reserve
 * cells).  fm_native_topk_paged is this call with res_mask = NULL, id_mode 0.
 *
 *   res_mask    NULL (every chunk of the listed pages is a candidate) or
 *               [ceil(Q / mask_group), mask_ld] uint32: chunk c = logical
 *               page * 64 + o of query qi is a candidate iff bit c & 31 of
 *               word c >> 5 of row qi / mask_group is set (words at or past
 *               mask_ld count as 0).  The Memory-Indexer bitmask
 *               (fm_memindex_score_mask's mask_out, one row per request) is
 *               this layout, with mask_group = layers per request.  A chunk
 *               that is not a candidate is never selected: fewer than k
 *               candidates -> all of them, padded with -1.
 *   mask_ld     words per mask row (>= 1 when res_mask is given)
 *   mask_group  consecutive queries sharing one mask row (>= 1)
 *   id_mode     0: idx_out holds logical chunk ids; 1: reserve cells
 *               page_phys * 64 + o (the pool row of the chunk).  The
 *               selection, its tie-break and its order are the same in both
 *               modes (by logical chunk id).
 * Other arguments, outputs and errors as fm_native_topk_paged (the same
 * workspace size); FM_ERR_INVALID_ARG also for a bad id_mode / mask_ld /
 * mask_group.
 */
fm_status fm_native_topk_paged_ex(const uint16_t* q, const float* w, const void* k_pool, int key_dtype,
                                  const float* k_scale, int64_t P, const int32_t* page_phys, const int32_t* page_logical,
                                  const int32_t* n_res, int Q, int R, int n_h, int d, int k,
                                  const uint32_t* res_mask, int64_t mask_ld, int mask_group, int id_mode,
                                  int32_t* idx_out, float* score_out, void* workspace, size_t workspace_bytes,
                                  fm_stream_t stream);

/*
 * Native paged top-k without a caller workspace.
 *
 * The pages have no counterpart of this entry point: it exists for callers
 * that cannot allocate device memory -- a serving engine that handed nearly
 * all of HBM to its KV-cache pool at start-up (a further cudaMalloc would fail
 * or fragment that pool), a decode loop that must not stall on the implicit
 * device synchronisation cudaMalloc/cudaFree may perform, or a plugin host that
 * gives its kernels no allocator.  It computes exactly what
 * fm_native_topk_paged computes for an E4M3 pool (key_dtype
 * FM_DTYPE_FP8_E4M3), with the same arguments minus key_dtype and the
 * workspace, and calls no allocating routine.
 *
 * Its scratch is a fixed FM_NOALLOC_SCRATCH_BYTES array inside the library's
 * device image: every GPU that loads the library holds it until the process
 * exits.  Sizes whose workspace (fm_native_topk_paged_workspace(Q, R)) exceeds
 * it are rejected with FM_ERR_INVALID_ARG before anything is enqueued (e.g.
 * R = 384 allows 136 queries per call).  Every call looks up the
 * array's device address (cudaGetSymbolAddress) with the calling thread's
 * current device, so the address stays right after a device reset; the first
 * call on a device also loads the library's device image there, so make that
 * first call before any stream capture.  All calls share the array and it
 * keeps the last call's contents (nothing in it needs to start at zero), so
 * calls that overlap on the GPU -- different streams or host threads -- race
 * on it: serialise them.
 */
#define FM_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
fm_status fm_native_topk_paged_noalloc(const uint16_t* q, const float* w, const uint8_t* k_pool,
                                       const float* k_scale, int64_t P, const int32_t* page_phys,
                                       const int32_t* page_logical, const int32_t* n_res, int Q, int R, int n_h,
                                       int d, int k, int32_t* idx_out, float* score_out, fm_stream_t stream);

/*
 * Prefill: dense indexer scores of T query tokens against S chunk keys under
 * the causal chunk limit, then top-k per query ([V4] sec. 3 CSA-1/2; chunk s
 * covers tokens ratio*s .. ratio*s + ratio-1, [V4] sec. 1/8).
 *
 *     Y[t,s] = sum_h w[t,h] * ReLU( sum_j q[t,h,j] * keys[s,j] ),
 * candidates of query t: s < min(S, floor(pos[t] / ratio)) (none if pos < 0).
 *
 *   q       [T, n_h, d] bf16, 16-byte aligned;  w [T, n_h] fp32
 *   pos     [T] int64 token positions
 *   keys    [S, d] bf16, 16-byte aligned
 *   T >= 0, S >= 0 (S < 2^31), ratio >= 1 (4 for c4), 1 <= k <= 1024
 *   idx_out [T, k] int32; score_out [T, k] fp32 or NULL
 *   workspace >= fm_index_prefill_workspace(T, S) bytes, 256-byte aligned
 */
size_t fm_index_prefill_workspace(int T, int64_t S);

/*
 * The prefill call's dense scores alone ([V4] sec. 3 CSA-1, the score the
 * CSA-2 top-512 ranks), for callers that select or inspect them themselves:
 *     logits_out[t, s] = Y[t,s]  for s < min(S, floor(pos[t] / ratio)),
 *                        -inf    otherwise.
 * Arguments as fm_index_prefill_topk; logits_out [T, S] fp32, row stride S,
 * 4-byte aligned (caller-owned; every element is written).  Two kernel
 * launches (the scores, then -inf past each token's limit), no workspace.
 */
fm_status fm_index_prefill_scores(const uint16_t* q, const float* w, const int64_t* pos, const uint16_t* keys,
                                  int T, int64_t S, int n_h, int d, int ratio, float* logits_out, fm_stream_t stream);
fm_status fm_index_prefill_topk(const uint16_t* q, const float* w, const int64_t* pos, const uint16_t* keys,
                                int T, int64_t S, int n_h, int d, int ratio, int k, int32_t* idx_out,
                                float* score_out, void* workspace, size_t workspace_bytes, fm_stream_t stream);

/*
 * Device status word of the current device: the OR of FM_DEVERR_* bits set by
 * kernels since the last reset.  Synchronises `stream` before reading.  When
 * reset != 0 the word is cleared after reading.  status_out is HOST memory.
 */
fm_status fm_device_status(uint32_t* status_out, int reset, fm_stream_t stream);

/*
 * The device status word as a status code: synchronises `stream`, reads the
 * word, clears it, and returns FM_OK when no bit was set,
 * FM_ERR_DEVICE_TIMEOUT when FM_DEVERR_TIMEOUT was set (a launch gave up: its
 * outputs are incomplete), otherwise FM_ERR_DEVICE_BOUNDS (page ids were
 * skipped; the outputs are those of the table without them).  fm_last_error
 * names the bits.  Kernels on other streams may set bits at any time: call it
 * where the caller's own work is known to be complete.
 */
fm_status fm_check_device_status(fm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FM_INDEX_H */
