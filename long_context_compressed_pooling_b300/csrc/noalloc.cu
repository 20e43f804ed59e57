// csa_index_topk_noalloc: the indexer + top-k call for callers that cannot allocate device
// memory. Its BF16 score scratch is a fixed array compiled into the library instead of a
// caller-provided workspace. See include/csa.h for the contract.
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/csa.h"
#include "kernels.h"

namespace {

// Score scratch shared by every call on a device: 8 MiB = 4,194,304 BF16 scores
// (B * Nq * E at most). Each device that loads the library holds it until the process exits.
constexpr size_t kNoAllocScoreBytes = size_t(8) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scores[kNoAllocScoreBytes];

constexpr int kMaxDevices = 64;
uint16_t* g_scores_on_device[kMaxDevices] = {};
std::mutex g_mu;

// Device address of the scratch array on the current device. In host code the array's name is
// only a host-side stand-in, so its address must come from cudaGetSymbolAddress, resolved once
// per device with that device current.
uint16_t* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scores_on_device[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scores) != cudaSuccess) return nullptr;
    g_scores_on_device[dev] = static_cast<uint16_t*>(p);
  }
  return g_scores_on_device[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" csa_status csa_index_topk_noalloc(const uint8_t* qi_codes, const uint8_t* qi_scales,
                                             const uint8_t* ki_codes, const uint8_t* ki_scales,
                                             int B, int Nq, int64_t q_pos0, int64_t E, int m,
                                             int H_I, int d_I, int k, int32_t* topk_idx,
                                             int32_t* topk_cnt, void* stream) {
  if (!qi_codes || !qi_scales || !ki_codes || !ki_scales || !topk_idx || !topk_cnt)
    return CSA_ERR_INVALID_ARG;
  if (!aligned16(qi_codes) || !aligned16(ki_codes) || !aligned16(ki_scales) ||
      !aligned16(topk_idx) || !aligned16(topk_cnt))
    return CSA_ERR_ALIGN;
  if (B < 1 || Nq < 1 || q_pos0 < 0 || E < 0 || m < 1 || k < 1) return CSA_ERR_INVALID_ARG;
  if (d_I != 32 && d_I != 64) return CSA_ERR_UNSUPPORTED;
  if (H_I != 1 && H_I != 2 && H_I != 4 && H_I != 8) return CSA_ERR_UNSUPPORTED;
  if ((uint64_t)B * (uint64_t)Nq * (uint64_t)E * 2u > kNoAllocScoreBytes)
    return CSA_ERR_WORKSPACE;  // more scores than the fixed scratch holds
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* scores = scratch_on_current_device();
  uint32_t* status = csa::device_status_word();
  if (!scores || !status) return CSA_ERR_CUDA;
  if (E > 0) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return CSA_ERR_CUDA;
    alignas(64) CUtensorMap map;
    const cuuint64_t row = (cuuint64_t)(d_I / 2);
    cuuint64_t dims[3] = {row, (cuuint64_t)E, (cuuint64_t)B};
    cuuint64_t strides[2] = {row, row * (cuuint64_t)E};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(ki_codes), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CSA_ERR_CUDA;
    const csa::IndexerPlan plan = csa::plan_indexer(B, Nq, E, H_I, d_I);
    if (csa::launch_indexer(&map, ki_codes, qi_codes, qi_scales, ki_scales, scores, B, Nq, q_pos0, E, m, H_I,
                            d_I, plan, status, st) != cudaSuccess)
      return CSA_ERR_CUDA;
  }
  return csa::launch_topk(scores, B, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, st) == cudaSuccess
             ? CSA_OK
             : CSA_ERR_CUDA;
}
