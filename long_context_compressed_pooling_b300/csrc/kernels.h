// Host-side launchers of the sm_103a kernels (internal to the library; the public C ABI is
// include/csa.h). Every launcher enqueues on `stream` and returns the launch's cudaError_t.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace csa {

// Launches `kern` with programmatic stream serialisation (the kernel may start while its
// predecessor on the stream finishes; every kernel of the library waits on griddepcontrol before
// touching data a predecessor wrote) and, when cluster_x > 1, as clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

constexpr int kNumSMs = 148;

// ---- paged heterogeneous KV cache (one layer; paged.cu has the layout) ------------------------
constexpr int kPageTokens = 4096;  // tokens per classical-cache page (a multiple of lcm(4, 128))
constexpr int kRingTokens = 256;   // raw tokens kept per sequence in the state cache
struct PagedLayout {
  int d, m, d_I;
  uint16_t* k_pool;                // [n_pages, kPageTokens / m, d] entries
  uint16_t* v_pool;
  uint8_t* ki_codes_pool;          // CSA: [n_pages, kPageTokens / m, d_I / 2] (null for HCA)
  uint8_t* ki_scales_pool;         // CSA: [n_pages, kPageTokens / m, d_I / 32]
  const int32_t* block_table;      // [B, max_blocks]: page of tokens [4096 i, 4096 (i + 1))
  int n_pages, max_blocks;
  uint16_t* ring_k;                // [B, kRingTokens, d] raw rows at slot (position % 256)
  uint16_t* ring_v;
  float* ring_logits;              // [B, kRingTokens]
  uint16_t* ring_xi;               // CSA: [B, kRingTokens, d_I] index-key rows (or null)
};
// Appends token t of every sequence to the state cache and compresses the block it closes.
cudaError_t launch_paged_append(const PagedLayout& L, int B, const uint16_t* k_new,
                                const uint16_t* v_new, const float* logit_new,
                                const uint16_t* xi_new, int64_t t, uint32_t* status,
                                cudaStream_t stream);

// The library's device status word on the current device (defined in abi.cu).
uint32_t* device_status_word();

// Failure injection for tests (csa_test_set_faults): the bounded-wait budget in SM cycles the
// kernels use, and a mask of producers (kFault* in common.cuh) that skip their work.
constexpr long long kWaitBudgetCyclesHost = 2000000000LL;  // equals kWaitBudgetCycles
struct FaultConfig {
  long long wait_budget;
  uint32_t skip_mask;
};
FaultConfig fault_config();

// ---- block pooling --------------------------------------------------------------------------
// The indexer's own compressed keys: pool index-key rows [B, N, d_I] of entries
// [j_begin, j_begin + n_entries) and convert them to MX FP4 (d_I in {32, 64, 128}, m <= 32).
cudaError_t launch_index_keys(const uint16_t* xi_raw, const float* logits, int B, int64_t N, int d_I,
                              int m, int64_t j_begin, int64_t n_entries, uint8_t* ki_codes,
                              uint8_t* ki_scales, cudaStream_t stream);
// MX FP4 conversion of bf16 rows [rows, d], d in {32, 64, 128}.
cudaError_t launch_mxfp4_quantize(const uint16_t* x, int64_t rows, int d, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t stream);
cudaError_t launch_compress(const uint16_t* k_raw, const uint16_t* v_raw, const float* logits,
                            int B, int64_t N, int d, int m, int64_t j_begin, int64_t n_entries,
                            uint16_t* k_cmp, uint16_t* v_cmp, cudaStream_t stream);

// ---- Lightning Indexer (tcgen05 FP4) ---------------------------------------------------------
struct IndexerPlan {
  int QN;        // queries per CTA
  int ncols;     // MMA N
  int G;         // tiles per MMA commit / epilogue pass
  int nacc;      // accumulator groups in tensor memory
  int n_groups;  // ceil(Nq / QN)
  int n_splits;  // entry-tile splits per (sequence, query group)
  int tmem_cols; // tensor-memory columns allocated per CTA
};
IndexerPlan plan_indexer(int B, int Nq, int64_t E, int H_I, int d_I, bool paged = false);
bool indexer_bulk_path(int H_I, int d_I, int64_t E, int Nq);
cudaError_t launch_indexer(const CUtensorMap* kmap, const uint8_t* ki_codes, const uint8_t* qi_codes,
                           const uint8_t* qi_scales, const uint8_t* ki_scales, uint16_t* scores,
                           int B, int Nq, int64_t q_pos0, int64_t E, int m, int H_I, int d_I,
                           const IndexerPlan& plan, uint32_t* status, cudaStream_t stream,
                           float* scores_f32 = nullptr, const PagedLayout* paged = nullptr,
                           int64_t keys_fresh_from = 0, bool q_fresh = true);
// keys_fresh_from / q_fresh: the index-key entries at or above keys_fresh_from, and (q_fresh)
// the index queries, may be the output of the kernel launched just before on the stream; the
// indexer reads them only after its grid-dependency wait. The defaults (everything may be
// fresh) are right for any caller that does not know its predecessor.

// ---- top-k over BF16 scores ------------------------------------------------------------------
// nonneg: every score is a non-negative BF16 value with zero stored as +0 (the indexer's
// output), so the selection uses the bit patterns as keys unchanged.
cudaError_t launch_topk(const uint16_t* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                        int k, int32_t* topk_idx, int32_t* topk_cnt, cudaStream_t stream,
                        bool nonneg = false);
// The same selection over FP32 scores [B, Nq, E] (rows of at most 16 x 32768 keys; longer rows
// return cudaErrorInvalidValue).
cudaError_t launch_topk_f32(const float* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                            int k, int32_t* topk_idx, int32_t* topk_cnt, cudaStream_t stream);

// ---- attention (CSA sparse / HCA dense) ------------------------------------------------------
struct AttendArgs {
  const uint16_t* q;
  const uint16_t* k_cmp;
  const uint16_t* v_cmp;
  const int32_t* topk_idx;  // null for HCA
  const int32_t* topk_cnt;  // null for HCA
  const uint16_t* k_raw;
  const uint16_t* v_raw;
  uint16_t* out;
  float* lse;
  int64_t E, N, q_pos0;
  int k, m, W, B, Nq, H, d;
  // Paged cache: entries through the block table, window rows from the ring (d = 128 only).
  const PagedLayout* paged = nullptr;
  // Dense attention only: entries [0, fresh_from) are inputs of this launch, and every kernel
  // before the one that precedes it on the stream has completed, so they may be read before
  // waiting for that predecessor; entries from fresh_from on may be its output. 0: wait first.
  int64_t fresh_from = 0;
};
int plan_attend_splits(int tokens, int H, int d, int64_t max_keys);
size_t attend_workspace_bytes(int tokens, int H, int d, int64_t max_keys);
// d = 128 runs the tcgen05 kernel (attend_tc.cu); d = 64 the tcgen05 kernel with several query
// tokens per CTA (attend_pk.cu) for prefill, the split-K mma.sync kernel (attend.cu) for decode.
cudaError_t launch_attend(const AttendArgs& a, int64_t max_keys, void* ws, uint32_t* status,
                          cudaStream_t stream);
cudaError_t launch_attend_pk(const AttendArgs& a, uint32_t* status, cudaStream_t stream);
int attend_tc_chunk_keys();
// n_splits CTAs per (token, 64-head group); cluster = 1 merges the splits through distributed
// shared memory (returns cudaErrorNotSupported if such a cluster cannot be scheduled), else the
// splits write ws_o / ws_ml for the merge kernel. n_splits = 1 (without a cluster) launches
// persistent CTAs, at most one per SM, each walking several (token, head group) items.
cudaError_t launch_attend_tc(const AttendArgs& a, int n_splits, int cluster, float* ws_o,
                             float* ws_ml, uint32_t* status, cudaStream_t stream);

// ---- entry-sharded selection and attention (shard.cu) ------------------------------------------
constexpr int kMaxShards = 16;
// cand_scores[b][j] = scores[b][sel[b][j]] for j < cnt[b], else 0.
cudaError_t launch_candidates(const uint16_t* scores, int B, int64_t E, const int32_t* sel,
                              const int32_t* cnt, int k, uint16_t* cand_scores, uint32_t* status,
                              cudaStream_t stream);
// The global top-k of S shards' candidates [S, B, k] (local indices; shard_base: host array of
// S first global indices), and each shard's part of it [S, B, k] (local indices).
cudaError_t launch_topk_merge(const uint16_t* cand_scores, const int32_t* cand_idx,
                              const int32_t* cand_cnt, const int64_t* shard_base, int B, int S,
                              int k, int32_t* topk_idx, int32_t* topk_cnt, int32_t* shard_idx,
                              int32_t* shard_cnt, cudaStream_t stream);
cudaError_t launch_lse_merge(const uint16_t* parts, const float* lse, int S, int64_t rows, int d,
                             uint16_t* out, float* lse_out, cudaStream_t stream);

// ---- batched row copies (stage.cu): a step's staged inputs into the layer buffers ----
constexpr int kMaxScatterCopies = 16;
struct ScatterCopy {
  void* dst;           // row r at dst + r * dst_stride
  const void* src;     // row r at src + r * row_bytes (rows packed)
  int64_t rows, row_bytes, dst_stride;
};
// n <= kMaxScatterCopies copies (validated by the caller) in one launch.
cudaError_t launch_scatter_rows(const ScatterCopy* copies, int n, cudaStream_t stream);

// ---- fused CSA decode step (decode.cu): indexer + top-k (+ sparse attention) in one launch ----
constexpr int kDecodeMaxCluster = 16;   // CTAs per sequence
constexpr int kDecodeMaxChunk = 16384;  // entries one CTA scores (BF16 scores kept on chip)
constexpr int kDecodeMaxKeys = 256;     // attention keys one CTA gathers
constexpr int kDecodeMaxSel = 2048;     // largest k
constexpr int kDecodeFusedChunk = 8192; // the planner takes the one-launch kernel up to this chunk
constexpr int kMaxDevicesDecode = 64;
struct DecodePlan {
  bool ok;
  int C, chunk, P;  // cluster size, entries per CTA, attention keys per CTA
};
struct DecodeArgs {
  const uint8_t* qi_codes;   // [B, H_I, 32] (one query per sequence, d_I = 64)
  const uint8_t* qi_scales;  // [B, H_I, 2]
  const uint8_t* ki_codes;   // [B, E, 32]
  const uint8_t* ki_scales;  // [B, E, 2]
  uint16_t* scores;          // optional [B, E] BF16 scores
  int32_t* topk_idx;         // [B, k]
  int32_t* topk_cnt;         // [B]
  int64_t E, t;              // entries, position of the query token
  int m, k, H_I, B;
  int64_t keys_fresh_from;   // as launch_indexer
  bool wait_first;           // true: the kernel before may write any input (queries included)
  bool attend;               // also the sparse attention (d = 128, H <= 64)
  int H, W;
  const uint16_t* q;         // [B, H, 128]
  uint16_t* k_cmp;           // written only for the pooled entries (below)
  uint16_t* v_cmp;           // [B, E, 128]
  const uint16_t* k_raw;
  const uint16_t* v_raw;     // [B, N, 128]
  uint16_t* out;             // [B, H, 128]
  float* lse;                // optional [B, H]
  int64_t N;
  // entries [pool_j0, pool_j1) pooled inside the launch (at most kDecodePoolMax per sequence;
  // pool_j1 == pool_j0: none), with csa_compress's arithmetic; k_cmp / v_cmp are written there
  const float* logits;
  int64_t pool_j0, pool_j1;
};
constexpr int kDecodePoolMax = 4;
// ok = false when the shape is outside the kernel's limits (E % 8 != 0, k > 2048, more than
// 16 x 16384 visible entries, more than 16 x 256 attention keys).
DecodePlan plan_decode(int B, int64_t E, int64_t n_vis, int k, int W, bool attend,
                       bool want_scores);
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& pl, uint32_t* status,
                          cudaStream_t stream);
// The decode kernel's indexer alone (no cluster, no selection) for rows too long for the
// one-launch step: BF16 scores of the visible entries into a.scores, each sequence split over
// `split` CTAs of `chunk` entries (plan_decode_scores: false when a CTA's share would exceed
// kDecodeMaxChunk, or E % 8 != 0).
bool plan_decode_scores(int B, int64_t E, int64_t n_vis, int* split, int* chunk);
cudaError_t launch_decode_scores(const DecodeArgs& a, int split, int chunk, uint32_t* status,
                                 cudaStream_t stream);

}  // namespace csa
