// Host-side launchers of the sm_103a kernels (internal to the library; the public C ABI is
// include/csa.h). Every launcher enqueues on `stream` and returns the launch's cudaError_t.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

constexpr int kNumSMs = 148;

// The library's device status word on the current device (defined in abi.cu).
uint32_t* device_status_word();

// ---- block pooling --------------------------------------------------------------------------
cudaError_t launch_compress(const uint16_t* k_raw, const uint16_t* v_raw, const float* logits,
                            int B, int64_t N, int d, int m, int64_t j_begin, int64_t n_entries,
                            uint16_t* k_cmp, uint16_t* v_cmp, cudaStream_t stream);

// ---- Lightning Indexer (tcgen05 FP4) ---------------------------------------------------------
struct IndexerPlan {
  int QN;        // queries per CTA
  int ncols;     // MMA N
  int n_groups;  // ceil(Nq / QN)
  int n_splits;  // entry-tile splits per (sequence, query group)
  int tmem_cols; // tensor-memory columns allocated per CTA
};
IndexerPlan plan_indexer(int B, int Nq, int64_t E, int H_I, int d_I);
cudaError_t launch_indexer(const CUtensorMap* kmap, const uint8_t* qi_codes,
                           const uint8_t* qi_scales, const uint8_t* ki_scales, uint16_t* scores,
                           int B, int Nq, int64_t q_pos0, int64_t E, int m, int H_I, int d_I,
                           const IndexerPlan& plan, uint32_t* status, cudaStream_t stream);

// ---- top-k over BF16 scores ------------------------------------------------------------------
cudaError_t launch_topk(const uint16_t* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
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
};
int plan_attend_splits(int tokens, int H, int64_t max_keys);
size_t attend_workspace_bytes(int tokens, int H, int d, int64_t max_keys);
cudaError_t launch_attend(const AttendArgs& a, int64_t max_keys, void* ws, uint32_t* status,
                          cudaStream_t stream);

}  // namespace csa
