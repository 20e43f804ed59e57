/*
 * csa.h -- C ABI of the B300 (sm_103a) CSA / HCA hybrid compressed attention library.
 *
 * The method (DeepSeek-V4 hybrid attention as described by the Lighthouse page "deep deepseek
 * v4 release", section 八.3, and the 9fzt.com DeepSeek-V4 summary, items 1 and 4):
 *   CSA  every m = 4 consecutive KV tokens are pooled into one compressed entry; a Lightning
 *        Indexer with an FP4 QK path scores the entries (scores rounded to BF16); a per-query
 *        top-k keeps k entries; attention runs over the kept entries plus a sliding window of
 *        n_win raw tokens.
 *   HCA  every m' = 128 tokens are pooled into one entry; attention is dense over all visible
 *        entries plus the same window.
 * The two layer types alternate along depth (elebank "DeepSeek-V4 explained", 模型創新 1).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers, row-major and contiguous, 16-byte aligned
 *     (per-row counts such as topk_cnt: 4-byte aligned).
 *     The caller owns every buffer; the library never allocates device memory on these paths.
 *   - bf16 values travel as uint16_t bit patterns. `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream). Every call is asynchronous on `stream`.
 *   - FP4 vectors are e2m1 codes packed two per byte, the low nibble holding the even element;
 *     each run of 32 elements has one UE8M0 scale byte s meaning 2^(s-127) (OCP MX v1.0).
 *   - Positions: the queries of a sequence sit at token positions q_pos0 .. q_pos0+Nq-1 of a
 *     context of N tokens (q_pos0 + Nq <= N). A query at position t sees compressed entry j iff
 *     (j+1)*m - 1 <= t, and the raw window tokens max(0, t-W+1) .. t. Entries and window tokens
 *     form one softmax (no de-duplication); logits are q.k with no extra scale.
 *   - Errors: arguments are validated before anything is launched and a CSA_ERR_* code is
 *     returned without side effects. A failed launch returns CSA_ERR_CUDA. Kernels never trap:
 *     an out-of-range top-k index, an unmapped page or an expired bounded wait is recorded
 *     in a device status word that csa_get_device_status() reads. Shapes the kernels do not
 *     implement return CSA_ERR_UNSUPPORTED (there is no fallback path).
 */
#ifndef CSA_B300_H
#define CSA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum csa_status {
  CSA_OK = 0,
  CSA_ERR_INVALID_ARG = 1,  /* null pointer, negative or zero size where one is required */
  CSA_ERR_SHAPE = 2,        /* sizes inconsistent with each other */
  CSA_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned */
  CSA_ERR_WORKSPACE = 4,    /* workspace pointer null or smaller than the *_workspace_size() */
  CSA_ERR_UNSUPPORTED = 5,  /* a shape outside the implemented set (see each call) */
  CSA_ERR_CUDA = 6,         /* a CUDA runtime call or kernel launch failed */
  CSA_ERR_DEVICE = 7        /* csa_get_device_status: a kernel recorded a fault (see below) */
} csa_status;

/* Device status bits (csa_get_device_status() returns CSA_ERR_DEVICE when any is set). */
#define CSA_DEVFLAG_BAD_INDEX 0x1u  /* a top-k index outside [0, E), a count above k/visible,
                                       or a paged cache's block-table entry naming no page */
#define CSA_DEVFLAG_TIMEOUT   0x2u  /* a bounded mbarrier wait expired; the kernel returned */

/* ----------------------------------------------------------------------------------------
 * csa_compress -- block pooling (CSA m=4, HCA m=128).
 * Lighthouse "deep deepseek v4 release" 八.3 (m = 4 / m' = 128 tokens into one entry);
 * the pooling operator is a softmax over the block's per-token logits:
 *   p_i = softmax_i(logits[jm+i]),  k_cmp[j] = sum_i p_i k_raw[jm+i],  v_cmp[j] likewise.
 *   k_raw, v_raw : [B, N, d] bf16          logits : [B, N] fp32
 *   k_cmp, v_cmp : [B, N/m, d] bf16 (entry cache, written in place)
 * Writes the entries j with tok_begin <= j*m and (j+1)*m <= tok_end; other entries are left
 * untouched. tok_begin must be a multiple of m; 0 <= tok_begin <= tok_end <= N.
 * Accumulation is fp32 (expf), entries are rounded to bf16 (round-to-nearest-even).
 * Supported: d in {64, 128, 256}, m a power of two in [1, 256]. k_cmp may equal v_cmp only
 * if k_raw equals v_raw.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_compress(const uint16_t* k_raw, const uint16_t* v_raw, const float* logits,
                        int B, int64_t N, int d, int m, int64_t tok_begin, int64_t tok_end,
                        uint16_t* k_cmp, uint16_t* v_cmp, void* stream);

/* ----------------------------------------------------------------------------------------
 * csa_compress_index_keys -- the Lightning Indexer's own compressed keys.
 * Lighthouse "deep deepseek v4 release" 八.7 lists them as a KV form of their own beside the
 * CSA / HCA entries; 9fzt.com item 4 puts the indexer's QK path in FP4. Pages give no
 * conversion rule; this library pools per-token index-key rows with the block pooling of
 * csa_compress (same softmax over the block's logits), rounds each pooled value to bf16
 * (round-to-nearest-even; a zero is +0) and converts every 32-element block to MX FP4 with the
 * OCP Microscaling Formats v1.0 rule (section 6.3): scale X = 2^(floor(log2 max|v|) - 2) as a
 * UE8M0 byte (0 for an all-zero block, exponent clamped to [-127, 127]), elements v / X rounded
 * to nearest-even on the E2M1 grid, magnitudes above 6 clamped to 6.
 *   xi_raw    : [B, N, d_I] bf16 index-key rows      logits : [B, N] fp32
 *   ki_codes  : [B, N/m, d_I/2] packed e2m1 (low nibble = even element), written in place
 *   ki_scales : [B, N/m, d_I/32] UE8M0
 * Writes entries j with tok_begin <= j*m and (j+1)*m <= tok_end, as csa_compress.
 * Supported: d_I in {32, 64, 128}, m a power of two in [1, 32]. xi_raw and ki_codes 16-byte
 * aligned. Inputs must be finite.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_compress_index_keys(const uint16_t* xi_raw, const float* logits, int B, int64_t N,
                                   int d_I, int m, int64_t tok_begin, int64_t tok_end,
                                   uint8_t* ki_codes, uint8_t* ki_scales, void* stream);

/* ----------------------------------------------------------------------------------------
 * csa_quantize_mxfp4 -- MX FP4 conversion of bf16 rows (the indexer's queries), the rule of
 * csa_compress_index_keys applied to each row as given (the sign of -0 is kept: code 8).
 *   x : [rows, d] bf16     codes : [rows, d/2] packed e2m1     scales : [rows, d/32] UE8M0
 * Supported: d in {32, 64, 128}; x and codes 16-byte aligned; finite inputs.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_quantize_mxfp4(const uint16_t* x, int64_t rows, int d, uint8_t* codes,
                              uint8_t* scales, void* stream);

/* ----------------------------------------------------------------------------------------
 * csa_index_topk -- Lightning Indexer scores + per-query top-k.
 * 9fzt.com DeepSeek-V4 summary item 4 (FP4 indexer QK path; index scores rounded from FP32 to
 * BF16), Lighthouse 八.3 (top-k over compressed entries), 八.7 (the indexer keeps its own
 * compressed keys).
 *   s[b,i,j] = bf16_rne( sum_h max(0, q_I[b,i,h] . k_I[b,j]) ) for visible j
 * with FP4 values times per-32 UE8M0 scales. When every scale byte lies in [123, 127] and
 * d_I <= 64, H_I <= 4, the fp32 sum is exact, so the bf16 scores are exact.
 *   qi_codes  [B, Nq, H_I, d_I/2] u8     qi_scales [B, Nq, H_I, d_I/32] u8
 *   ki_codes  [B, E, d_I/2] u8           ki_scales [B, E, d_I/32] u8
 *   topk_idx  [B, Nq, k] int32 out: the min(k, visible) entries with the largest score, ties
 *             to the lower index, sorted ascending, padded with -1
 *   topk_cnt  [B, Nq] int32 out: min(k, visible)
 *   scores    optional [B, Nq, E] bf16 out (NULL: kept in the workspace). Only visible
 *             entries are written.
 * The scores are computed on the tensor cores (tcgen05 FP4 MMA, fp32 accumulators in tensor
 * memory). Supported: d_I in {32, 64}, H_I in {1, 2, 4, 8}, k >= 1, scale bytes in [1, 254].
 * Workspace: csa_index_topk_workspace_size().
 * ---------------------------------------------------------------------------------------- */
csa_status csa_index_topk(const uint8_t* qi_codes, const uint8_t* qi_scales,
                          const uint8_t* ki_codes, const uint8_t* ki_scales,
                          int B, int Nq, int64_t q_pos0, int64_t E, int m, int H_I, int d_I,
                          int k, int32_t* topk_idx, int32_t* topk_cnt, uint16_t* scores,
                          void* ws, size_t ws_bytes, void* stream);
size_t csa_index_topk_workspace_size(int B, int Nq, int64_t E, int k, int scores_given);

/* ----------------------------------------------------------------------------------------
 * csa_index_topk_noalloc -- csa_index_topk for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment variant of the call above.
 * Some callers hold no allocator of their own: a plugin or kernel-library host whose device
 * memory is owned by a framework pool, code running under a memory budget or inside a region
 * where cudaMalloc's implicit synchronisation is not acceptable, or a C caller that only has its
 * input and output pointers. This entry point takes the same inputs and outputs as
 * csa_index_topk but no workspace: its BF16 score scratch is a fixed 8 MiB array inside the
 * library (every GPU that loads the library keeps it until the process exits), so
 * B * Nq * E must not exceed 4,194,304 scores; larger calls return CSA_ERR_WORKSPACE.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 * The first call on each device resolves the array's device address (cudaGetSymbolAddress with
 * that device current); make that first call before any stream capture.
 * Every call on a device shares the one array, which keeps the last call's scores: calls whose
 * execution overlaps on the GPU (other streams, or concurrent host threads) race on it and must
 * be serialised by the caller.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_index_topk_noalloc(const uint8_t* qi_codes, const uint8_t* qi_scales,
                                  const uint8_t* ki_codes, const uint8_t* ki_scales,
                                  int B, int Nq, int64_t q_pos0, int64_t E, int m, int H_I,
                                  int d_I, int k, int32_t* topk_idx, int32_t* topk_cnt,
                                  void* stream);

/* ----------------------------------------------------------------------------------------
 * csa_topk -- the top-k selector alone, over caller-provided BF16 scores [B, Nq, E]
 * (9fzt.com item 4: the selector works on BF16 index scores). Same outputs and tie rule as
 * csa_index_topk. -0 counts as +0; NaN scores are not supported.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_topk(const uint16_t* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                    int k, int32_t* topk_idx, int32_t* topk_cnt,
                    void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------------------------
 * csa_index_scores -- the Lightning Indexer alone: BF16 scores [B, Nq, E] as csa_index_topk
 * computes them and, when scores_f32 is not NULL, the exact FP32 scores [B, Nq, E] they are
 * rounded from (9fzt.com item 4: the scores were FP32 before being reduced to BF16; every
 * FP32 score here is exact, so the BF16 score is its round-to-nearest-even). Only visible
 * entries (those csa_index_topk scores for each query) are written. Same inputs and limits as
 * csa_index_topk; scores and scores_f32 16-byte aligned.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_index_scores(const uint8_t* qi_codes, const uint8_t* qi_scales,
                            const uint8_t* ki_codes, const uint8_t* ki_scales, int B, int Nq,
                            int64_t q_pos0, int64_t E, int m, int H_I, int d_I, uint16_t* scores,
                            float* scores_f32, void* stream);

/* ----------------------------------------------------------------------------------------
 * csa_topk_f32 -- the selector of csa_topk over FP32 scores [B, Nq, E]: the selection the
 * pages' BF16 scores replace (9fzt.com item 4 reports the BF16 selector 2x faster). Same
 * order, tie rule, outputs and padding as csa_topk (-0 counts as +0; NaN not supported).
 * Rows of at most 16 x 32768 visible entries (CSA_ERR_UNSUPPORTED beyond).
 * ---------------------------------------------------------------------------------------- */
csa_status csa_topk_f32(const float* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                        int k, int32_t* topk_idx, int32_t* topk_cnt, void* stream);
size_t csa_topk_workspace_size(int B, int Nq, int64_t E, int k);

/* ----------------------------------------------------------------------------------------
 * csa_attend -- CSA attention over the selected entries plus the sliding window.
 * Lighthouse 八.3 (sparse attention over the top-k compressed blocks, plus a sliding-window
 * branch of n_win raw tokens).
 *   out[b,i,h] = sum_n softmax_n(q[b,i,h] . key_n) value_n over
 *   {k_cmp[b, topk_idx[b,i,r]] : r < topk_cnt[b,i]}  +  {k_raw[b,u] : u in window(t)}
 *   q [B, Nq, H, d] bf16 (1/sqrt(d) already folded in), k_cmp/v_cmp [B, E, d] bf16,
 *   k_raw/v_raw [B, N, d] bf16, out [B, Nq, H, d] bf16, lse optional [B, Nq, H] fp32
 *   (natural log of the softmax denominator; -inf and out = 0 for an empty key set).
 * Indices outside [0, E) are skipped and flagged (CSA_DEVFLAG_BAD_INDEX).
 * Supported: d in {64, 128}, 1 <= H <= 128, 0 <= W, 0 <= k.
 * Workspace: csa_attend_workspace_size() (split-K partials for small batches).
 * ---------------------------------------------------------------------------------------- */
csa_status csa_attend(const uint16_t* q, const uint16_t* k_cmp, const uint16_t* v_cmp, int64_t E,
                      const int32_t* topk_idx, const int32_t* topk_cnt, int k,
                      const uint16_t* k_raw, const uint16_t* v_raw, int64_t N, int W,
                      int B, int Nq, int64_t q_pos0, int H, int d,
                      uint16_t* out, float* lse, void* ws, size_t ws_bytes, void* stream);
size_t csa_attend_workspace_size(int B, int Nq, int H, int d, int k, int W);

/* ----------------------------------------------------------------------------------------
 * hca_attend -- HCA dense attention over every visible entry plus the sliding window.
 * Lighthouse 八.3 (m' = 128, dense attention, no top-k). Same tensors as csa_attend without
 * the top-k lists; m is the block size that defines entry visibility.
 * ---------------------------------------------------------------------------------------- */
csa_status hca_attend(const uint16_t* q, const uint16_t* k_cmp, const uint16_t* v_cmp, int64_t E,
                      int m, const uint16_t* k_raw, const uint16_t* v_raw, int64_t N, int W,
                      int B, int Nq, int64_t q_pos0, int H, int d,
                      uint16_t* out, float* lse, void* ws, size_t ws_bytes, void* stream);
size_t hca_attend_workspace_size(int B, int Nq, int H, int d, int64_t E, int m, int W);

/* ----------------------------------------------------------------------------------------
 * csa_hca_layer_pair -- one CSA layer followed by one HCA layer (they alternate along depth:
 * Lighthouse 八.3, elebank 模型創新 1). Each layer: compress the blocks of tokens
 * [compress_begin, N) into its entry cache, then (CSA) index + top-k and attend, or (HCA)
 * attend densely. The two layers get independent inputs; either descriptor may be NULL.
 * Fields follow the single calls above.
 * Concurrency: with both layers present, the HCA layer runs on a side stream owned by the
 * library (one per device, created on the first call that is not being captured into a CUDA
 * graph), forked from `stream` and joined back into it with events; work enqueued on `stream`
 * afterwards sees both layers complete. Without the side stream (a graph capture before any
 * eager call) everything runs on `stream`.
 * Workspace: csa_hca_layer_pair_workspace_size() = a CSA region (scores, then the CSA
 * attention's split-K partials) followed by a disjoint HCA region.
 * ---------------------------------------------------------------------------------------- */
typedef struct csa_layer_desc {
  const uint16_t* q;            /* [B, Nq, H, d] */
  const uint16_t* k_raw;        /* [B, N, d] */
  const uint16_t* v_raw;        /* [B, N, d] */
  const float* logits;          /* [B, N] */
  const uint8_t* qi_codes;      /* [B, Nq, H_I, d_I/2] */
  const uint8_t* qi_scales;     /* [B, Nq, H_I, d_I/32] */
  const uint8_t* ki_codes;      /* [B, N/m, d_I/2] (written for new entries when xi_raw set) */
  const uint8_t* ki_scales;     /* [B, N/m, d_I/32] (likewise) */
  uint16_t* k_cmp;              /* [B, N/m, d] entry cache (in/out) */
  uint16_t* v_cmp;              /* [B, N/m, d] entry cache (in/out) */
  uint16_t* out;                /* [B, Nq, H, d] */
  float* lse;                   /* optional [B, Nq, H] */
  int32_t* topk_idx;            /* [B, Nq, k] */
  int32_t* topk_cnt;            /* [B, Nq] */
  uint16_t* scores;             /* optional [B, Nq, N/m] */
  int B, Nq, H, d, m, W, k, H_I, d_I;
  int64_t N, q_pos0, compress_begin;
  /* optional [B, N, d_I] bf16 index-key rows: when set, the layer also writes the indexer keys
   * of the entries it compresses (csa_compress_index_keys over [compress_begin, N)) before
   * scoring; when NULL, ki_codes / ki_scales are inputs. */
  const uint16_t* xi_raw;
} csa_layer_desc;

typedef struct hca_layer_desc {
  const uint16_t* q;
  const uint16_t* k_raw;
  const uint16_t* v_raw;
  const float* logits;
  uint16_t* k_cmp;              /* [B, N/m, d] */
  uint16_t* v_cmp;
  uint16_t* out;
  float* lse;                   /* optional */
  int B, Nq, H, d, m, W;
  int64_t N, q_pos0, compress_begin;
} hca_layer_desc;

csa_status csa_hca_layer_pair(const csa_layer_desc* csa, const hca_layer_desc* hca,
                              void* ws, size_t ws_bytes, void* stream);

/* ----------------------------------------------------------------------------------------
 * Paged heterogeneous KV cache with incremental decode-time compression.
 * Lighthouse "deep deepseek v4 release" 八.7: the cache is split into a state cache (the
 * sliding window and the tail of tokens not yet compressed) and a classical cache (the
 * compressed entries), with cache blocks aligned to lcm(m, m') tokens. Layout here (one layer):
 *   classical cache  pools of pages; page p holds the entries of CSA_PAGE_TOKENS = 4096
 *                    consecutive tokens of one sequence (4096 / m entries, and for CSA their
 *                    index keys); block_table[b * max_blocks + i] is the page of tokens
 *                    [4096 i, 4096 (i + 1)) of sequence b. 4096 is a multiple of
 *                    lcm(4, 128) = 128, so a block of m tokens never straddles pages.
 *   state cache      rings of the last CSA_RING_TOKENS = 256 raw tokens per sequence: the token
 *                    at position p sits in slot p % 256 of ring_k, ring_v, ring_logits (and, for
 *                    CSA, ring_xi: the index-key rows the indexer's keys are pooled from).
 * csa_paged_decode_step appends token N of every sequence (all sequences hold N tokens before
 * the call) to the state cache; when N closes a block (N % m == m - 1) it pools the block from
 * the ring into its page, with csa_compress's arithmetic (and, for CSA with xi rows, the index
 * key as csa_compress_index_keys); then it decodes the new token against the cache exactly as
 * the flat path does at t = N: CSA scores the (N + 1) / m visible entries with the indexer,
 * selects the top-k and attends to the selected entries plus the window; HCA attends densely.
 * Supported: d = 128, W <= 128; CSA: m a power of two <= 32, d_I = 64, H_I <= 4; HCA: m a
 * power of two <= 128. Every pointer 16-byte aligned (ring_logits, logit_new: 4). Pages must
 * be mapped (block_table entries in [0, n_pages)) for every block up to token N; an unmapped
 * page is flagged in the device status word and its keys are left out. The caller owns the
 * pools, rings and block table; the call writes the new token's ring slots, at most one entry
 * per layer (plus its index key), out, lse, topk_idx, topk_cnt and the workspace.
 * ---------------------------------------------------------------------------------------- */
#define CSA_PAGE_TOKENS 4096
#define CSA_RING_TOKENS 256

typedef struct csa_paged_layer {
  int kind;                     /* 0: CSA (indexer, top-k, sparse attention), 1: HCA (dense) */
  int B, H, d, m, W, k, H_I, d_I;
  int64_t N;                    /* tokens per sequence before this step */
  uint16_t* k_pool;             /* [n_pages, 4096 / m, d] bf16 entries */
  uint16_t* v_pool;
  uint8_t* ki_codes_pool;       /* CSA: [n_pages, 4096 / m, d_I / 2] packed e2m1 */
  uint8_t* ki_scales_pool;      /* CSA: [n_pages, 4096 / m, d_I / 32] UE8M0 */
  const int32_t* block_table;   /* [B, max_blocks] */
  int n_pages, max_blocks;
  uint16_t* ring_k;             /* [B, 256, d] bf16 */
  uint16_t* ring_v;
  float* ring_logits;           /* [B, 256] */
  uint16_t* ring_xi;            /* CSA: [B, 256, d_I] bf16, or NULL (keys written elsewhere) */
  const uint16_t* k_new;        /* [B, d] the appended token's K row */
  const uint16_t* v_new;        /* [B, d] */
  const float* logit_new;       /* [B] its pooling logit */
  const uint16_t* xi_new;       /* CSA: [B, d_I] its index-key row (with ring_xi) */
  const uint16_t* q;            /* [B, H, d] the new token's queries */
  const uint8_t* qi_codes;      /* CSA: [B, H_I, d_I / 2] */
  const uint8_t* qi_scales;     /* CSA: [B, H_I, d_I / 32] */
  uint16_t* out;                /* [B, H, d] */
  float* lse;                   /* optional [B, H] */
  int32_t* topk_idx;            /* CSA: [B, k] */
  int32_t* topk_cnt;            /* CSA: [B] */
} csa_paged_layer;

size_t csa_paged_decode_workspace_size(const csa_paged_layer* layer);
csa_status csa_paged_decode_step(const csa_paged_layer* layer, void* ws, size_t ws_bytes,
                                 void* stream);

/* csa_paged_layer_pair -- one paged decode step of a CSA layer (kind 0) and an HCA layer
 * (kind 1), the HCA layer on a library-owned side stream beside the CSA layer (joined before
 * the call's later work on `stream`, as in csa_hca_layer_pair). The workspace holds the two
 * layers' regions one after the other. */
size_t csa_paged_layer_pair_workspace_size(const csa_paged_layer* csa,
                                           const csa_paged_layer* hca);
csa_status csa_paged_layer_pair(const csa_paged_layer* csa, const csa_paged_layer* hca,
                                void* ws, size_t ws_bytes, void* stream);
size_t csa_hca_layer_pair_workspace_size(const csa_layer_desc* csa, const hca_layer_desc* hca);

/* ----------------------------------------------------------------------------------------
 * Status.
 * csa_get_device_status synchronises `stream`, reads the device status word of the current
 * device and returns CSA_OK, CSA_ERR_DEVICE (flags in *flags_out when non-NULL) or
 * CSA_ERR_CUDA; reset != 0 clears the word afterwards.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_get_device_status(void* stream, int reset, uint32_t* flags_out);

/* ----------------------------------------------------------------------------------------
 * Entry-sharded decode: the compressed entries of each sequence split over S shards (GPUs, or
 * slices of one GPU's cache); shard s holds entries [shard_base[s], shard_base[s] + E_s). The
 * pages' 1M-token context (9fzt.com DeepSeek-V4 summary, item 1) with the CSA selection and
 * attention of Lighthouse 八.3. Every entry of the global top-k is among its own shard's top-k,
 * so merging the shards' candidates gives exactly the unsharded selection (score descending,
 * ties to the lower global index); each shard then attends to its part of the selection (one
 * shard also to the window) and the partial outputs merge by their log-sum-exp.
 *
 * csa_shard_candidates -- one shard's top-k candidates of one query per sequence: csa_index_topk
 *   over the shard's entries (ki_codes / ki_scales point at the shard's first entry, E = E_s,
 *   q_pos0 = t - shard_base * m so that visibility is the global one), returning the local
 *   indices (cand_idx [B, k], ascending, -1 pad), their BF16 scores (cand_scores [B, k], 0 pad)
 *   and counts (cand_cnt [B]). Workspace: csa_shard_candidates_workspace_size (the shard's
 *   scores). Same limits as csa_index_topk.
 * csa_topk_merge -- the global top-k of S shards' candidates, shard-major: cand_scores and
 *   cand_idx [S, B, k], cand_cnt [S, B] (each shard's csa_shard_candidates outputs stacked, k of
 *   every shard equal); shard_base: HOST array of S ascending first global indices.
 *   topk_idx [B, k] global indices ascending, -1 pad; topk_cnt [B] = min(k, candidates);
 *   shard_idx [S, B, k] the local indices of each shard's part of the selection (ascending, -1
 *   pad); shard_cnt [S, B]. Supported: S <= 16, k <= 2048.
 * csa_lse_merge -- out[r] = sum_s e^(lse_s[r] - L) parts[s][r] with L = log sum_s e^(lse_s[r])
 *   (a shard with lse = -inf has weight 0; all -inf gives out = 0, lse = -inf).
 *   parts [S, rows, d] bf16 (each shard's normalised output, as csa_attend writes it),
 *   parts_lse [S, rows] fp32, out [rows, d] bf16, lse optional [rows]. d a multiple of 8.
 * ---------------------------------------------------------------------------------------- */
csa_status csa_shard_candidates(const uint8_t* qi_codes, const uint8_t* qi_scales,
                                const uint8_t* ki_codes, const uint8_t* ki_scales, int B,
                                int64_t q_pos0, int64_t E, int m, int H_I, int d_I, int k,
                                int32_t* cand_idx, uint16_t* cand_scores, int32_t* cand_cnt,
                                void* ws, size_t ws_bytes, void* stream);
size_t csa_shard_candidates_workspace_size(int B, int64_t E, int k);
csa_status csa_topk_merge(const uint16_t* cand_scores, const int32_t* cand_idx,
                          const int32_t* cand_cnt, const int64_t* shard_base, int B, int S, int k,
                          int32_t* topk_idx, int32_t* topk_cnt, int32_t* shard_idx,
                          int32_t* shard_cnt, void* stream);
csa_status csa_lse_merge(const uint16_t* parts, const float* parts_lse, int S, int64_t rows, int d,
                         uint16_t* out, float* lse, void* stream);

/* ----------------------------------------------------------------------------------------
 * csa_test_set_faults -- failure injection for tests of the device-side failure detection
 * (no counterpart on the pages). Every wait of a kernel on data another warp or copy produces
 * is bounded; on expiry the kernel records CSA_DEVFLAG_TIMEOUT, releases what it holds and
 * returns. wait_budget_cycles > 0 replaces the bound (about 2e9 SM cycles, one second) for
 * every later launch of a kernel that honours it; <= 0 restores it. skip_mask names producers
 * that skip their work on later launches, so that the waits depending on them run out:
 *   CSA_FAULT_SKIP_KEY_COPIES  the indexer's copy warp issues no key copies (csa_index_topk,
 *                              csa_index_scores, the CSA layer of csa_hca_layer_pair); the
 *                              call's top-k outputs are then unspecified, but in range.
 * Returns CSA_ERR_INVALID_ARG for unknown bits. The settings are process-wide; a test restores
 * them with csa_test_set_faults(0, 0) and clears the status word with csa_get_device_status.
 * After a timeout, attention launches skip their work until the status word is cleared.
 * ---------------------------------------------------------------------------------------- */
#define CSA_FAULT_SKIP_KEY_COPIES 0x1u
#define CSA_FAULT_ALL             0x1u
csa_status csa_test_set_faults(long long wait_budget_cycles, uint32_t skip_mask);

/* ----------------------------------------------------------------------------------------
 * Batched row copies on the device (data movement of a serving loop; no counterpart on the
 * pages). A step's new inputs can travel host-to-device as one packed upload into a staging
 * buffer; this call then places them into the layer buffers in one launch. Copy i moves
 * rows rows of row_bytes bytes each from src (rows packed: row r at src + r * row_bytes) to dst
 * (row r at dst + r * dst_stride). dst and src are device pointers; descs is a host array of
 * n <= CSA_MAX_COPIES descriptors, read before the call returns. Copies must not overlap one
 * another or their sources. Rows move 16 bytes at a time when a copy's pointers, row_bytes and
 * dst_stride are multiples of 16. The launch signals no dependent kernel before it completes,
 * so a library call enqueued after it on the same stream reads the placed rows.
 * Errors: CSA_ERR_INVALID_ARG for descs == NULL with n > 0, n < 0 or n > CSA_MAX_COPIES,
 * negative rows / row_bytes, dst_stride < row_bytes with rows > 1, or a null pointer in a
 * copy that moves bytes; CSA_ERR_CUDA if the launch fails.
 * ---------------------------------------------------------------------------------------- */
#define CSA_MAX_COPIES 16
typedef struct csa_copy_desc {
  void* dst;
  const void* src;
  int64_t rows;
  int64_t row_bytes;
  int64_t dst_stride;
} csa_copy_desc;
csa_status csa_scatter_rows(const csa_copy_desc* descs, int n, void* stream);

/* ----------------------------------------------------------------------------------------
 * Per-kernel timing (tracing aid; no counterpart on the pages). While enabled, every kernel
 * launch of the library is bracketed by two CUDA events recorded on its launch stream.
 * csa_profiler_collect synchronises those events and returns, per kernel name, the number of
 * launches and their summed device time; reset != 0 clears the records. At most 32768 launches
 * are recorded between resets; later ones are not timed.
 * ---------------------------------------------------------------------------------------- */
typedef struct csa_kernel_time {
  char name[32];
  int launches;
  double total_ms;
} csa_kernel_time;
csa_status csa_profiler_enable(int on);
csa_status csa_profiler_collect(csa_kernel_time* out, int max_entries, int* n_entries, int reset);
const char* csa_status_string(csa_status s);
int csa_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA_B300_H */
