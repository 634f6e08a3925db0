/*
 * tq.h -- C ABI of the TurboQuant KV-cache hot path for NVIDIA GB300 (sm_103a).
 *
 * Keys are stored as TurboQuant_prod records and values as TurboQuant_mse
 * records in fixed 16-token pages; decode attention scores the query directly
 * against the packed codes.  Sources (page title, section):
 *   [Design study]   "TurboQuant Family Design Study for CPU and Browser WASM
 *                    KV Caches"
 *   [Reconstruction] "Mathematical Reconstruction, Lineage, and Accuracy Limits
 *                    of TurboQuant and TurboVec"
 *   [README]         "TurboQuant: KV Cache Compression for LLM Inference"
 *
 * Conventions for every entry point
 *   - Ownership: the caller owns every buffer.  No call allocates memory;
 *     scratch memory for decode is a caller-provided workspace.
 *   - Device pointers are marked [device]; host pointers [host].
 *   - Asynchrony: calls that take a cudaStream_t only enqueue work on that
 *     stream and never synchronise, except tq_check_device_error.
 *   - Errors: arguments are checked on the host before any launch; a failed
 *     check returns a tq_status != TQ_OK, launches nothing, and sets a
 *     thread-local message readable with tq_last_error().  A launch failure
 *     returns TQ_ERR_CUDA.  Data-dependent faults found on the device (a page
 *     index outside the pool, a sequence longer than its block table) never
 *     trap: the kernel skips the access and sets a device error word, read and
 *     cleared by tq_check_device_error().
 *   - Layout of one vector: a vector is (token, kv head); index n = token *
 *     n_kv_heads + head; input rows are d contiguous elements.
 *   - Bit planes: coordinate j sits at bit (j mod 32) of 32-bit word j / 32.
 *     A b-bit code is stored sign-magnitude: plane 0 = 1 iff
 *     idx >= 2^(b-1); planes 1..b-1 = magnitude m (LSB first), with
 *     m = idx - 2^(b-1) on the non-negative side and 2^(b-1)-1-idx otherwise.
 *     The QJL sketch is one plane, bit = 1 iff (S r)_j >= 0.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tq_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or combination */
  TQ_ERR_UNSUPPORTED = 2,    /* valid but not built: d, bit width, page size */
  TQ_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
  TQ_ERR_NO_CONVERGENCE = 4, /* Lloyd-Max iteration cap reached */
  TQ_ERR_CAPACITY = 5,       /* workspace or pool too small */
  TQ_ERR_DEVICE_CHECK = 6    /* the device error word was set (see below) */
} tq_status;

typedef enum { TQ_DENSE = 0, TQ_FWHT = 1 } tq_transform_kind;
typedef enum { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;
typedef enum { TQ_ROLE_KEY_ROT = 0, TQ_ROLE_VALUE_ROT = 1, TQ_ROLE_QJL = 2, TQ_ROLE_QJL_SIGNS = 3 } tq_role;

/* Device error word bits (tq_check_device_error). */
#define TQ_DEVERR_PAGE_INDEX 0x1u   /* block-table entry outside [0, n_pages) */
#define TQ_DEVERR_SEQ_LEN    0x2u   /* seq_len beyond block table + window   */
#define TQ_DEVERR_SLOT       0x4u   /* slot_mapping entry outside the pool   */
#define TQ_DEVERR_TIMEOUT    0x8u   /* a bounded wait on a TMA copy ran out  */
#define TQ_DEVERR_CODEBOOK   0x10u  /* two code boundaries in one cell of the
                                       quantize kernels' code table (their
                                       codes are then unreliable; not expected:
                                       the host picks the table's scale)     */

#define TQ_PAGE_SIZE 16
#define TQ_MAX_BITS 4
#define TQ_MAX_GQA 8

/*
 * tq_build_codebook -- Lloyd-Max codebook for one rotated coordinate.
 * [Reconstruction] §5 Steps 2-4: continuous k-means on the marginal of one
 * coordinate of a uniformly rotated unit vector in R^d (density
 * proportional to (1-x^2)^((d-3)/2) on [-1, 1]).  Runs on the host, in double.
 *   d            4 <= d <= 4096
 *   bits         1..4 (2^bits levels)
 *   centroids    [host] out, float[2^bits], ascending, RMS scale (sqrt(d) * c)
 *   boundaries   [host] out, float[2^bits - 1], float32 midpoints of
 *                neighbouring centroids; the decision rule is
 *                idx = #{i : z >= boundaries[i]} with z = sqrt(d) * (Pi u)_j
 *   mse_unit     [host] out, nullable: E||u - u_hat||^2 for unit u
 * Returns TQ_ERR_NO_CONVERGENCE if 100000 iterations do not converge.
 */
tq_status tq_build_codebook(int d, int bits, float* centroids, float* boundaries, double* mse_unit);

/*
 * tq_build_transform -- the seeded random draws of the method, on the host.
 * [Reconstruction] §5 Step 2 (dense rotation via QR of a Gaussian matrix),
 * §6 (QJL matrix S, i.i.d. N(0,1)), §9 and §13 (Rademacher signs + fast
 * Walsh-Hadamard); [Design study] §Dense and structured transform comparison.
 * Generator: SplitMix64 from state seed ^ mix((layer << 24) | (head << 8) | role).
 *   kind=TQ_DENSE, role 0/1: out = float[d*d] row-major Haar rotation Pi
 *                            (y = Pi u); Householder QR, column signs fixed.
 *   kind=TQ_FWHT,  role 0/1: out = float[d] Rademacher signs sigma; the
 *                            rotation is Pi u = H (sigma * u) / sqrt(d).
 *   role 2 (either kind):    out = float[d*d] row-major QJL matrix S.
 *   role 3 (either kind):    out = float[d] Rademacher signs sigma_S of the
 *                            structured QJL matrix S = H diag(sigma_S).
 *   out [host]. d must be a power of two for TQ_FWHT; 2 <= d <= 4096.
 */
tq_status tq_build_transform(tq_transform_kind kind, int d, uint64_t seed, int layer, int head,
                             int role, float* out);

/*
 * Key corrections on top of the Lloyd-Max code ([Reconstruction] §6 QJL;
 * §10 / §12.2 EDEN's unbiased scale, 2.75x lower 1-bit variance than QJL;
 * §12 item 2 and §13 step 6 TurboVec's length-renormalized correction, one
 * scalar per key, norm / <y, y_hat>, said there to restore unbiasedness).
 * EDEN and RENORM keep the scale in the record slot QJL uses for gamma and
 * spend no bit on a sketch.  With the norm stored in its own field both store
 * the same number, s = ||y||^2 / <y, y_hat> = 1 / <y, y_hat> (y the rotated
 * unit key, y_hat its centroids); the two names are kept so that a caller can
 * ask for either method by name.
 */
typedef enum { TQ_KEY_MSE = 0, TQ_KEY_QJL = 1, TQ_KEY_EDEN = 2, TQ_KEY_RENORM = 3 } tq_key_correction;

/*
 * Per-layer parameters.  Transforms are per KV head.  The codebooks are held
 * by value (from tq_build_codebook); entries beyond 2^bits are ignored.
 */
typedef struct {
  int d;           /* head dimension: 128 or 256 (power of two, multiple of 32) */
  int n_kv_heads;  /* Hkv >= 1 */
  int n_q_heads;   /* Hq, a multiple of Hkv with Hq / Hkv <= 8 */
  int page_size;   /* must be 16 */
  int window;      /* W >= 0 recent tokens kept float16 */
  int key_bits;    /* MSE bits of the key code, 1..4 */
  int key_qjl;     /* key correction, a tq_key_correction: TQ_KEY_QJL = TurboQuant_prod (QJL sign
                      sketch of the residual, gamma = ||r||); TQ_KEY_MSE = code only; TQ_KEY_EDEN /
                      TQ_KEY_RENORM = code plus one float scale s per key (EDEN's unbiased
                      ||y||^2 / <y, y_hat>; TurboVec's norm / <y, y_hat> divided by the stored
                      norm, the same number), score n s <q', y_hat> */
  int value_bits;  /* 1..4 */
  tq_transform_kind kind;
  const float* k_rot;  /* [device] [Hkv][d*d] (dense) or [Hkv][d] signs (FWHT) */
  const float* v_rot;  /* [device] same shape as k_rot                        */
  const float* qjl_s;  /* [device] [Hkv][d*d] QJL matrices ([Hkv][d] signs with qjl_structured);
                          NULL unless key_qjl == TQ_KEY_QJL */
  float k_centroids[16], k_bounds[16];
  float v_centroids[16], v_bounds[16];
  /* Length of the key, value, query and output vectors the caller passes;
   * 0 means d.  A head size that is not a power of two (a multiple of 8 with
   * d/2 < head_dim < d, e.g. 80 or 96 with d = 128, 160 with d = 256) is
   * zero-padded to d inside the kernels for the transforms and the codes, and
   * outputs keep head_dim coordinates ([Design study] §Dense and structured
   * transform comparison: temporary zero-padding during append and query
   * transform).  Codes, signs and the float16 window rows keep d
   * coordinates (the window's tail stays zero). */
  int head_dim;
  /* Mixed-channel key rate ([Design study] §Packed format and complete bit
   * accounting: fractional nominal rates by channel allocation, fixed offsets,
   * no decoder state).  0: every rotated coordinate takes key_bits bits.
   * 1: coordinates 0 .. d/2-1 take key_bits + 1 bits with the k_hi_* book
   * (a (key_bits+1)-bit tq_build_codebook), the rest key_bits bits with the
   * k_* book, e.g. key_bits = 3 for the 3.5 bits-per-channel key mode.
   * Needs key_bits <= 3 and key_qjl != TQ_KEY_QJL. */
  int key_split;
  float k_hi_centroids[16], k_hi_bounds[16];
  /* Key norms in the pages ([Design study] §Packed format, "u8 log-norm").
   * 0: float32.  1: one byte per token-head, code 0 for a zero vector, else
   * code = 1 + clamp(floor(t + 1/2), 0, 254) with
   * t = (log2 n - key_norm_log2_lo) / step, step = (hi - lo) / 254, decoded
   * as 2^(lo + (code - 1) step).  lo < hi, both finite; the flat
   * tq_quantize_keys output keeps float32 norms. */
  int key_norm_u8;
  float key_norm_log2_lo, key_norm_log2_hi;
  /* Structured QJL matrix ([Design study] §Candidate key and value
   * algorithms: the structured key arm with a residual QJL stage done in the
   * transform domain).  0: qjl_s holds [Hkv][d*d] i.i.d. N(0,1) matrices.
   * 1: qjl_s holds [Hkv][d] signs sigma_S (tq_build_transform role 3) and
   * S = H diag(sigma_S), H the unnormalised Sylvester Walsh-Hadamard matrix
   * (entries +-1, S S^T = d I); S r and S q' are computed with the fast
   * transform, the estimator keeps sqrt(pi/2)/d.  Needs key_qjl == TQ_KEY_QJL. */
  int qjl_structured;
  /* KIVI-like control arm ([Design study] §Candidate key and value
   * algorithms, arm 3: per-channel keys, per-token values, float16 recent
   * window).  1: asymmetric min-max integer codes of key_bits / value_bits
   * bits (2 or 4) in place of the TurboQuant records; a key group is one
   * channel over a page's 16 tokens, a value group one token over its d
   * channels; zero = float16(min), scale = float16((max - min) / (2^b - 1))
   * formed in float32; code = clamp(floor((x - zero) / scale + 1/2)), 0 where
   * the scale is 0.  No rotation or sketch (k_rot, v_rot, qjl_s unused; kind
   * ignored); key_qjl, key_split, key_norm_u8, qjl_structured must be 0;
   * head_dim == d; window >= 1 (pages are written whole: at a window flush,
   * or by page-aligned direct appends).  Flat tq_quantize_* do not apply. */
  int kivi;
} tq_layer_params;

/*
 * tq_quantize_keys -- TurboQuant_prod of n_vec key vectors (flat output).
 * [Reconstruction] §5 Steps 1-5 and §6: n = ||k||; y = Pi k / n; code of
 * z = sqrt(d) y; residual r = y - c[idx]/sqrt(d) in the rotated basis;
 * gamma = ||r||; QJL signs of S r.  If n < 1e-7 the record is norm 0,
 * gamma 0, codes of z = 0, all signs +1 ([Reconstruction] §11 item 2, §13).
 *   k           [device] [n_vec][head_dim] in dtype (vector n uses head n % Hkv);
 *               16-byte aligned
 *   code_planes [device] out, uint32 [n_vec][key_bits][d/32]; with key_split,
 *               uint32 [n_vec][key_bits * d/32 + d/64]: the key_bits planes over
 *               all coordinates, then the top plane of coordinates 0 .. d/2-1
 *   sign_planes [device] out, uint32 [n_vec][d/32]; NULL unless key_qjl == TQ_KEY_QJL
 *   norms       [device] out, float [n_vec]
 *   rnorms      [device] out, float [n_vec]: gamma (QJL) or the scale s (EDEN, RENORM); NULL iff MSE only
 * n_vec may be 0 (no launch).
 */
tq_status tq_quantize_keys(const tq_layer_params* p, const void* k, tq_dtype dtype, int64_t n_vec,
                           uint32_t* code_planes, uint32_t* sign_planes, float* norms, float* rnorms,
                           tq_stream_t stream);

/*
 * tq_quantize_values -- TurboQuant_mse of n_vec value vectors (flat output).
 * [Reconstruction] §5; [Design study] §Candidate key and value algorithms
 * (value path: MSE-oriented codec, no QJL residual).
 *   v           [device] [n_vec][head_dim] in dtype (vector n uses head n % Hkv)
 *   code_planes [device] out, uint32 [n_vec][value_bits][d/32]
 *   norms       [device] out, float [n_vec]
 */
tq_status tq_quantize_values(const tq_layer_params* p, const void* v, tq_dtype dtype, int64_t n_vec,
                             uint32_t* code_planes, float* norms, tq_stream_t stream);

/*
 * The paged cache of one layer ([Design study] §Packed format; §Paging,
 * lifecycle).  Page pool: [n_pages][Hkv][sub-block]; the sub-block of one
 * (page, kv head) holds 16 tokens, in this order:
 *   key norms          float [16]               (uint8 [16] with key_norm_u8)
 *   key residual norms float [16]              (key_qjl != 0: gamma or the scale s)
 *   key code planes    uint32 [key_bits][16][d/32]   token-major
 *   key top plane      uint32 [16][d/64]       (key_split only: coordinates < d/2)
 *   key sign plane     uint32 [16][d/32]       (key_qjl == TQ_KEY_QJL only)
 *   value norms        float [16]
 *   value code planes  uint16 [value_bits][d]  coordinate-major: bit t of
 *                      entry (plane, j) is that plane's bit of token t at j
 * (16 x the per-token record bytes; see tq_subblock_bytes).
 * KIVI arm (kivi = 1): key scales float16 [d], key zeros float16 [d], key
 * codes uint32 [16][d key_bits / 32] (code j of a token at bits
 * (j b) mod 32 of word (j b) / 32), value scales float16 [16], value zeros
 * float16 [16], value codes uint32 [16][d value_bits / 32].
 * Token position p of sequence b, p < n_compressed[b], lives in page
 * block_table[b][p / 16], slot p % 16.  Positions n_compressed[b] ..
 * seq_len[b]-1 are the float16 window; position p lives at ring slot
 * p mod (window + 16) of win_k / win_v.
 */
typedef struct {
  void* page_pool;            /* [device] 16-byte aligned                        */
  int64_t n_pages;
  const int32_t* block_table; /* [device] [batch][max_pages_per_seq]             */
  int max_pages_per_seq;
  int32_t* seq_len;           /* [device] [batch] tokens held (read/written)     */
  int32_t* n_compressed;      /* [device] [batch] tokens held in pages           */
  void* win_k;                /* [device] float16 [batch][Hkv][window+16][d], or NULL if window == 0 */
  void* win_v;                /* [device] same                                   */
  int batch;
} tq_cache;

/*
 * tq_prefill_cache -- fill every sequence of a cache with its first n_tok
 * tokens, applying the window rule of this page format in the library
 * ([Design study] §Packed format "Recent tokens", §Paging): with a window
 * W > 0 the
 *   n_c = 16 * floor(max(0, n_tok - W) / 16)
 * oldest tokens are quantized into their pages (position p of sequence b into
 * page block_table[b][p / 16], slot p % 16; whole pages, so the KIVI arm is
 * served too); without a window n_c = n_tok (the last page may be partly
 * filled, as decode-step appends leave it).  The remaining n_tok - n_c
 * (W .. W + 15 once n_tok >= W) are
 * written to the float16 window ring (position p at ring slot p mod (W + 16),
 * rows zero-padded past head_dim), and seq_len[b] = n_tok,
 * n_compressed[b] = n_c.  Decode-step appends (tq_append_page without a slot
 * mapping) continue from that state.
 *   k, v    [device] [batch][n_tok][Hkv][head_dim] in dtype, 16-byte aligned
 *   n_tok   tokens per sequence, >= 0
 * The sequences' previous contents are overwritten.  TQ_ERR_CAPACITY if n_c
 * needs more than max_pages_per_seq pages.  Page ids outside the pool set
 * TQ_DEVERR_SLOT in the device error word (those tokens are skipped).
 */
tq_status tq_prefill_cache(const tq_layer_params* p, tq_cache* cache, const void* k, const void* v,
                           tq_dtype dtype, int n_tok, tq_stream_t stream);

/* Bytes of one (page, kv head) sub-block; 0 for invalid parameters. */
size_t tq_subblock_bytes(const tq_layer_params* p);

/*
 * tq_append_page -- quantize new tokens into the paged cache.
 * [Design study] §Append cost ("the append path runs once per new decode
 * token"), §Packed format ("Recent tokens" window), §Paging.
 *   k, v       [device] [n_tok][Hkv][head_dim] in dtype
 *   slot_mapping == NULL (decode step): n_tok must equal cache->batch and
 *     token b is the next token of sequence b.  With window W > 0 it is
 *     written to the float16 ring; when the window then holds W + 16 tokens
 *     the oldest 16 are quantized (from their float16 values) into page
 *     block_table[b][n_compressed[b] / 16] and n_compressed[b] += 16.  With
 *     W == 0 it is quantized directly into slot seq_len[b] of its page.
 *     seq_len[b] and n_compressed[b] are updated on the device.
 *   slot_mapping != NULL (direct): [device] int64 [n_tok]; token t is
 *     quantized into pool slot slot_mapping[t] = page * 16 + slot for every
 *     KV head (negative entries are skipped).  Counters are not touched.
 */
tq_status tq_append_page(const tq_layer_params* p, tq_cache* cache, const void* k, const void* v,
                         tq_dtype dtype, int64_t n_tok, const int64_t* slot_mapping,
                         tq_stream_t stream);

/*
 * Workspace bytes for tq_decode_attention with the same (batch, max_ctx,
 * n_splits) arguments (n_splits = 0: automatic choice).
 */
size_t tq_decode_workspace_size(const tq_layer_params* p, int batch, int max_ctx, int n_splits);

/*
 * tq_decode_attention -- one decode query per sequence over the paged cache.
 * [Design study] §Transform placement (score against packed keys in the
 * rotated basis, q^T k = (T q)^T (T k)); §CPU and WASM kernel design
 * ("Decode-time key scan", "Decode-time value scan", FP32 accumulators,
 * inverse value transform once per head); [Reconstruction] §6 estimator.
 * For query head h (KV head g = h / (Hq / Hkv)):
 *   compressed token i:  l_i = scale * n_i * ( <Pi_g q, C_k[idx_i]> / sqrt(d)
 *                              + sqrt(pi/2)/d * gamma_i * <S_g Pi_g q, 2 s_i - 1> )
 *   window token i:      l_i = scale * <q, k_i>
 *   out = ( Pi_v^T sum_c p_i m_i C_v[vidx_i] / sqrt(d) + sum_w p_i v_i ),
 *   p = softmax(l) over all seq_len[b] tokens; lse = log sum exp(l).
 *   q        [device] [batch][Hq][head_dim] in dtype
 *   scale    softmax scale (usually 1/sqrt(d))
 *   out      [device] out, float [batch][Hq][head_dim]
 *   lse      [device] out, nullable, float [batch][Hq]
 *   scores   [device] out, nullable, float [batch][Hq][max_ctx]: every l_i
 *            at its token position (for inspection; costs extra stores)
 *   workspace [device] scratch of tq_decode_workspace_size bytes, 256-byte
 *            aligned; contents need not be initialised
 *   max_ctx  upper bound on every seq_len[b] (sizes the split-K grid)
 * A sequence with seq_len 0 gets out = 0 and lse = -inf.  batch <= 65535 and
 * batch * G <= 262140 (TQ_ERR_INVALID_ARG otherwise; the workspace size is then 0).
 */
tq_status tq_decode_attention(const tq_layer_params* p, const tq_cache* cache, const void* q,
                              tq_dtype dtype, float scale, float* out, float* lse, float* scores,
                              void* workspace, size_t workspace_bytes, int max_ctx, int n_splits,
                              tq_stream_t stream);

/*
 * tq_decode_attention_static -- tq_decode_attention without a workspace
 * argument, for callers that cannot allocate device memory (for example a
 * host runtime whose memory is all pre-planned, or code running where
 * cudaMalloc is forbidden or would stall).  The pages this library follows
 * have no counterpart to it; it is a convenience of this library.
 * The scratch lives in a fixed array inside the library, TQ_STATIC_SCRATCH_BYTES
 * large, which every GPU that loads the library keeps for the life of the
 * process.  Same arguments, results and errors as tq_decode_attention; a
 * configuration whose workspace (tq_decode_workspace_size) exceeds the array
 * returns TQ_ERR_CAPACITY and launches nothing.  Nothing is allocated.
 *   - The first call on each device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process: after cudaDeviceReset
 *     (or anything else that destroys the device's primary context) it no
 *     longer refers to the array, so a process that resets a device must not
 *     call this entry point on that device again.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (other streams, other host threads) race and corrupt each other's
 *     scratch.  Serialise them on one stream.  The array keeps the last call's
 *     contents; decode writes every scratch byte it reads, so nothing needs
 *     clearing between calls.
 */
#define TQ_STATIC_SCRATCH_BYTES (16u << 20)
tq_status tq_decode_attention_static(const tq_layer_params* p, const tq_cache* cache, const void* q,
                                     tq_dtype dtype, float scale, float* out, float* lse, float* scores,
                                     int max_ctx, int n_splits, tq_stream_t stream);

/*
 * tq_prefill_attention -- attention of a prefill chunk over the compressed
 * cache ([Design study] §Transform placement and §Packed format: the chunk's
 * queries are scored against the packed pages, not a decoded history; the
 * second workload next to decode).  The chunk's n_query tokens are the last
 * n_query tokens already appended to every sequence: query i of sequence b
 * sits at position p = seq_len[b] - n_query + i and attends causally to the
 * cached positions 0 .. p (compressed pages and the float16 window), with the
 * same score and output rules as tq_decode_attention.  Each query is a
 * virtual decode sequence of visible length p + 1 over its sequence's block
 * table and window ring.  For TurboQuant_prod keys (QJL sketch, 2 or 3 code
 * bits, no mixed-channel rate or byte norms) with values of 2..4 bits the
 * compressed pages are scored for 16 (query, head) rows of the chunk per page
 * pass (query tiles); other layers run the decode pipeline over the virtual
 * sequences.  The workspace size accounts for either.
 *   q         [device] [batch][n_query][Hq][head_dim] in dtype
 *   out       [device] out, float [batch][n_query][Hq][head_dim]
 *   lse       [device] out, float [batch][n_query][Hq] (nullable)
 *   workspace [device] 256-byte aligned, >= tq_prefill_workspace_size bytes
 *   max_ctx   upper bound of seq_len over the batch
 * seq_len[b] < n_query sets TQ_DEVERR_SEQ_LEN (those queries see the tokens
 * that exist).  batch * n_query <= 65535 and batch * n_query * G <= 262140
 * (TQ_ERR_INVALID_ARG otherwise; the workspace size is then 0).
 */
size_t tq_prefill_workspace_size(const tq_layer_params* p, int batch, int n_query, int max_ctx);
tq_status tq_prefill_attention(const tq_layer_params* p, const tq_cache* cache, int n_query, const void* q,
                               tq_dtype dtype, float scale, float* out, float* lse, void* workspace,
                               size_t workspace_bytes, int max_ctx, tq_stream_t stream);

/* Synchronises the stream, reads and clears the device error word.
 * Returns TQ_ERR_DEVICE_CHECK if any bit was set (bits in *bits_out, nullable). */
tq_status tq_check_device_error(tq_stream_t stream, uint32_t* bits_out);

/* Message for the last failed call on this thread ("" if none). */
const char* tq_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H_ */
