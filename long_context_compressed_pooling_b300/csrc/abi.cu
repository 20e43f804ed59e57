// extern "C" entry points of include/csa.h: argument validation, launch planning, TMA
// descriptor encoding and the CSA/HCA layer-pair driver. No entry point allocates device
// memory; scratch lives in the caller's workspace.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/csa.h"
#include "kernels.h"

using namespace csa;

namespace {

// Device status word (CSA_DEVFLAG_*), one per device that loads the library.
__device__ uint32_t g_device_status;

constexpr int kMaxDevices = 64;
uint32_t* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;

uint32_t* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
  }
  return g_status_ptr[dev];
}

// Side stream of the layer-pair driver, one per device, created on the first call that is not
// being captured into a CUDA graph (creating streams during a capture is not allowed). The HCA
// layer runs on it, joined back with an event; without it (a capture before any eager call) the
// driver runs everything on the caller's stream.
struct SideStreams {
  cudaStream_t s[2];
  cudaEvent_t ev[3];
};
SideStreams* g_side[kMaxDevices] = {};
bool g_side_failed[kMaxDevices] = {};

SideStreams* side_streams(cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_side[dev] != nullptr || g_side_failed[dev]) return g_side[dev];
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
    return nullptr;  // try again on an eager call
  SideStreams* ss = new SideStreams();
  bool ok = true;
  for (int i = 0; i < 2; ++i)
    ok = ok && cudaStreamCreateWithFlags(&ss->s[i], cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; i < 3; ++i)
    ok = ok && cudaEventCreateWithFlags(&ss->ev[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    (void)cudaGetLastError();
    delete ss;
    g_side_failed[dev] = true;
    return nullptr;
  }
  g_side[dev] = ss;
  return ss;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// per-row counts are read and written one int32 at a time: 4-byte alignment is enough
bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

csa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- validation of each call's arguments (no CUDA call is made before these pass) ----------
csa_status check_compress(const uint16_t* k_raw, const uint16_t* v_raw, const float* logits,
                          int B, int64_t N, int d, int m, int64_t tok_begin, int64_t tok_end,
                          uint16_t* k_cmp, uint16_t* v_cmp) {
  if (!k_raw || !v_raw || !logits || !k_cmp || !v_cmp) return CSA_ERR_INVALID_ARG;
  if (!al16(k_raw) || !al16(v_raw) || !al16(k_cmp) || !al16(v_cmp) || (uintptr_t)logits % 4)
    return CSA_ERR_ALIGN;
  if (B < 1 || N < 1 || m < 1) return CSA_ERR_INVALID_ARG;
  if (tok_begin < 0 || tok_end < tok_begin || tok_end > N || tok_begin % m != 0)
    return CSA_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return CSA_ERR_UNSUPPORTED;
  if (m > 256 || (m & (m - 1)) != 0) return CSA_ERR_UNSUPPORTED;
  if (k_cmp == v_cmp && k_raw != v_raw) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

csa_status check_index_inputs(const uint8_t* qi_codes, const uint8_t* qi_scales,
                              const uint8_t* ki_codes, const uint8_t* ki_scales, int B, int Nq,
                              int64_t q_pos0, int64_t E, int m, int H_I, int d_I,
                              const uint16_t* scores) {
  if (!qi_codes || !qi_scales || !ki_codes || !ki_scales) return CSA_ERR_INVALID_ARG;
  if (!al16(qi_codes) || !al16(ki_codes) || !al16(ki_scales) || (scores && !al16(scores)))
    return CSA_ERR_ALIGN;
  if (B < 1 || Nq < 1 || q_pos0 < 0 || E < 0 || m < 1) return CSA_ERR_INVALID_ARG;
  if (d_I != 32 && d_I != 64) return CSA_ERR_UNSUPPORTED;
  if (H_I != 1 && H_I != 2 && H_I != 4 && H_I != 8) return CSA_ERR_UNSUPPORTED;
  if (E > (int64_t)1 << 31 || (int64_t)B * Nq > ((int64_t)1 << 31) - 1) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

csa_status check_index(const uint8_t* qi_codes, const uint8_t* qi_scales,
                       const uint8_t* ki_codes, const uint8_t* ki_scales, int B, int Nq,
                       int64_t q_pos0, int64_t E, int m, int H_I, int d_I, int k,
                       const int32_t* topk_idx, const int32_t* topk_cnt, const uint16_t* scores) {
  csa_status s = check_index_inputs(qi_codes, qi_scales, ki_codes, ki_scales, B, Nq, q_pos0, E, m,
                                    H_I, d_I, scores);
  if (s != CSA_OK) return s;
  if (!topk_idx || !topk_cnt || k < 1) return CSA_ERR_INVALID_ARG;
  if (!al16(topk_idx) || !al4(topk_cnt)) return CSA_ERR_ALIGN;
  return CSA_OK;
}

csa_status check_topk(const uint16_t* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                      int k, const int32_t* topk_idx, const int32_t* topk_cnt) {
  if (!scores || !topk_idx || !topk_cnt) return CSA_ERR_INVALID_ARG;
  if (!al16(scores) || !al16(topk_idx) || !al4(topk_cnt)) return CSA_ERR_ALIGN;
  if (B < 1 || Nq < 1 || q_pos0 < 0 || E < 0 || m < 1 || k < 1) return CSA_ERR_INVALID_ARG;
  if ((int64_t)B * Nq > ((int64_t)1 << 31) - 1) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

csa_status check_attend(const uint16_t* q, const uint16_t* k_cmp, const uint16_t* v_cmp,
                        int64_t E, const uint16_t* k_raw, const uint16_t* v_raw, int64_t N, int W,
                        int B, int Nq, int64_t q_pos0, int H, int d, const uint16_t* out,
                        const float* lse) {
  if (!q || !k_cmp || !v_cmp || !k_raw || !v_raw || !out) return CSA_ERR_INVALID_ARG;
  if (!al16(q) || !al16(k_cmp) || !al16(v_cmp) || !al16(k_raw) || !al16(v_raw) || !al16(out) ||
      (lse && !al16(lse)))
    return CSA_ERR_ALIGN;
  if (B < 1 || Nq < 1 || H < 1 || N < 1 || W < 0 || E < 0 || q_pos0 < 0)
    return CSA_ERR_INVALID_ARG;
  if (q_pos0 + Nq > N) return CSA_ERR_SHAPE;
  if (d != 64 && d != 128) return CSA_ERR_UNSUPPORTED;
  if (H > 1024 || (int64_t)B * Nq > 65535LL * 32768LL) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

csa_status check_index_keys(const uint16_t* xi_raw, const float* logits, int B, int64_t N,
                            int d_I, int m, int64_t tok_begin, int64_t tok_end,
                            const uint8_t* ki_codes, const uint8_t* ki_scales) {
  if (!xi_raw || !logits || !ki_codes || !ki_scales) return CSA_ERR_INVALID_ARG;
  if (!al16(xi_raw) || !al16(ki_codes) || (uintptr_t)logits % 4) return CSA_ERR_ALIGN;
  if (B < 1 || N < 1 || m < 1) return CSA_ERR_INVALID_ARG;
  if (tok_begin < 0 || tok_end < tok_begin || tok_end > N || tok_begin % m != 0)
    return CSA_ERR_SHAPE;
  if (d_I != 32 && d_I != 64 && d_I != 128) return CSA_ERR_UNSUPPORTED;
  if (m > 32 || (m & (m - 1)) != 0) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}

// ---- internal runners (arguments already validated) -----------------------------------------
// What the indexer may read before its grid-dependency wait (kernels.h, launch_indexer). The
// default, for callers that do not know the kernel enqueued before them: nothing.
// Entries [j0, j1) of every sequence to pool (csa_compress's arithmetic) inside the scoring
// launch of a decode-shaped indexer call, instead of in a launch of their own.
struct PoolRange {
  const uint16_t* k_raw;
  const uint16_t* v_raw;
  const float* logits;
  uint16_t* k_cmp;
  uint16_t* v_cmp;
  int64_t N, j0, j1;
};

struct Freshness {
  int64_t keys_from = 0;
  bool queries = true;
  // optional: pool these entries inside the launch when the decode kernel scores (sets *pooled)
  const PoolRange* pool = nullptr;
  bool* pooled = nullptr;
};

void set_pool(DecodeArgs& a, const Freshness& fr) {
  if (!fr.pool) return;
  a.k_raw = fr.pool->k_raw;
  a.v_raw = fr.pool->v_raw;
  a.logits = fr.pool->logits;
  a.k_cmp = fr.pool->k_cmp;
  a.v_cmp = fr.pool->v_cmp;
  a.N = fr.pool->N;
  a.pool_j0 = fr.pool->j0;
  a.pool_j1 = fr.pool->j1;
  if (fr.pooled) *fr.pooled = true;
}

csa_status run_indexer(const uint8_t* qi_codes, const uint8_t* qi_scales, const uint8_t* ki_codes,
                       const uint8_t* ki_scales, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                       int H_I, int d_I, uint16_t* sc, float* scores_f32, cudaStream_t st,
                       const PagedLayout* paged = nullptr, Freshness fr = Freshness());

// The fused decode kernel (decode.cu) serves one query per sequence with 64-element index keys
// of at most 4 heads; its plan decides whether the rest of the shape fits.
bool decode_indexer_fits(int Nq, int H_I, int d_I) { return Nq == 1 && d_I == 64 && H_I <= 4; }

csa_status run_index_topk(const uint8_t* qi_codes, const uint8_t* qi_scales,
                          const uint8_t* ki_codes, const uint8_t* ki_scales, int B, int Nq,
                          int64_t q_pos0, int64_t E, int m, int H_I, int d_I, int k,
                          int32_t* topk_idx, int32_t* topk_cnt, uint16_t* scores, void* ws,
                          cudaStream_t st, Freshness fr = Freshness()) {
  if (decode_indexer_fits(Nq, H_I, d_I)) {
    const int64_t nv = std::max<int64_t>(0, std::min<int64_t>(E, (q_pos0 + 1) / m));
    const DecodePlan pl = plan_decode(B, E, nv, k, 0, false, scores != nullptr);
    if (pl.ok) {
      uint32_t* status = status_word();
      if (!status) return CSA_ERR_CUDA;
      DecodeArgs a{};
      a.qi_codes = qi_codes;
      a.qi_scales = qi_scales;
      a.ki_codes = ki_codes;
      a.ki_scales = ki_scales;
      a.scores = scores;
      a.topk_idx = topk_idx;
      a.topk_cnt = topk_cnt;
      a.E = E;
      a.t = q_pos0;
      a.m = m;
      a.k = k;
      a.H_I = H_I;
      a.B = B;
      a.keys_fresh_from = fr.keys_from;
      a.wait_first = fr.queries;
      a.attend = false;
      set_pool(a, fr);
      return from_cuda(launch_decode(a, pl, status, st));
    }
  }
  uint16_t* sc = scores ? scores : static_cast<uint16_t*>(ws);
  csa_status s = run_indexer(qi_codes, qi_scales, ki_codes, ki_scales, B, Nq, q_pos0, E, m, H_I,
                             d_I, sc, nullptr, st, nullptr, fr);
  if (s != CSA_OK) return s;
  return from_cuda(launch_topk(sc, B, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, st, true));
}

// The indexer alone: BF16 scores (and, when scores_f32 is set, the exact FP32 scores).
csa_status run_indexer(const uint8_t* qi_codes, const uint8_t* qi_scales, const uint8_t* ki_codes,
                       const uint8_t* ki_scales, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                       int H_I, int d_I, uint16_t* sc, float* scores_f32, cudaStream_t st,
                       const PagedLayout* paged, Freshness fr) {
  if (E > 0 && !paged && !scores_f32 && decode_indexer_fits(Nq, H_I, d_I)) {
    // one query per sequence: the decode kernel's indexer spread over the whole GPU
    const int64_t nv = std::max<int64_t>(0, std::min<int64_t>(E, (q_pos0 + 1) / m));
    int split = 0, chunk = 0;
    if (plan_decode_scores(B, E, nv, &split, &chunk)) {
      uint32_t* status = status_word();
      if (!status) return CSA_ERR_CUDA;
      DecodeArgs a{};
      a.qi_codes = qi_codes;
      a.qi_scales = qi_scales;
      a.ki_codes = ki_codes;
      a.ki_scales = ki_scales;
      a.scores = sc;
      a.E = E;
      a.t = q_pos0;
      a.m = m;
      a.k = 1;
      a.H_I = H_I;
      a.B = B;
      a.keys_fresh_from = fr.keys_from;
      a.wait_first = fr.queries;
      set_pool(a, fr);
      return from_cuda(launch_decode_scores(a, split, chunk, status, st));
    }
  }
  if (E > 0) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return CSA_ERR_CUDA;
    uint32_t* status = status_word();
    if (!status) return CSA_ERR_CUDA;
    alignas(64) CUtensorMap map;
    const cuuint64_t row = (cuuint64_t)(d_I / 2);
    // paged keys: one flat run of pool rows (the copies then go through the block table)
    const cuuint64_t rows = paged ? (cuuint64_t)paged->n_pages * (kPageTokens / m) : (cuuint64_t)E;
    cuuint64_t dims[3] = {row, rows, paged ? (cuuint64_t)1 : (cuuint64_t)B};
    cuuint64_t strides[2] = {row, row * rows};
    cuuint32_t box[3] = {32, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(ki_codes), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return CSA_ERR_CUDA;
    const IndexerPlan plan = plan_indexer(B, Nq, E, H_I, d_I, paged != nullptr);
    cudaError_t e = launch_indexer(&map, ki_codes, qi_codes, qi_scales, ki_scales, sc, B, Nq, q_pos0, E, m,
                                   H_I, d_I, plan, status, st, scores_f32, paged, fr.keys_from,
                                   fr.queries);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
  }
  return CSA_OK;
}

size_t index_ws_bytes(int B, int Nq, int64_t E, int scores_given) {
  return scores_given ? 0 : round_up((size_t)B * Nq * (size_t)E * 2, 256);
}

int64_t hca_max_keys(int64_t E, int m, int64_t N, int W) {
  const int64_t vis = N / m < E ? N / m : E;
  return vis + W;
}

}  // namespace

namespace {
// Failure injection (csa_test_set_faults); read at every launch of a kernel that honours it.
std::atomic<long long> g_wait_budget{0};
std::atomic<uint32_t> g_fault_mask{0};
}  // namespace

namespace csa {
// The library's device status word on the current device (null if it cannot be resolved).
uint32_t* device_status_word() { return status_word(); }

FaultConfig fault_config() {
  FaultConfig f;
  const long long b = g_wait_budget.load();
  f.wait_budget = b > 0 ? b : kWaitBudgetCyclesHost;
  f.skip_mask = g_fault_mask.load();
  return f;
}
}  // namespace csa

namespace {
size_t pair_csa_ws(const csa_layer_desc* c) {
  if (!c) return 0;
  const int64_t E = c->N / (c->m > 0 ? c->m : 1);
  const size_t a = index_ws_bytes(c->B, c->Nq, E, c->scores != nullptr);
  const size_t b = attend_workspace_bytes(c->B * c->Nq, c->H, c->d, (int64_t)c->k + c->W);
  return round_up(a > b ? a : b, 256);
}
size_t pair_hca_ws(const hca_layer_desc* h) {
  if (!h) return 0;
  const int64_t E = h->N / (h->m > 0 ? h->m : 1);
  return round_up(attend_workspace_bytes(h->B * h->Nq, h->H, h->d, E + h->W), 256);
}
size_t paged_ws(const csa_paged_layer* L) {
  if (!L || L->m < 1) return 0;
  const int64_t E = (L->N + 1) / L->m;
  const size_t a = L->kind == 0 ? index_ws_bytes(L->B, 1, E, 0) : 0;
  const int64_t keys = (L->kind == 0 ? (int64_t)L->k : E) + L->W;
  const size_t b = attend_workspace_bytes(L->B, L->H, L->d, keys);
  return round_up(a > b ? a : b, 256);
}

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

csa_status check_paged(const csa_paged_layer* L) {
  if (!L) return CSA_ERR_INVALID_ARG;
  const bool csa_kind = L->kind == 0;
  if (L->kind != 0 && L->kind != 1) return CSA_ERR_INVALID_ARG;
  if (!L->k_pool || !L->v_pool || !L->block_table || !L->ring_k || !L->ring_v ||
      !L->ring_logits || !L->k_new || !L->v_new || !L->logit_new || !L->q || !L->out)
    return CSA_ERR_INVALID_ARG;
  if (csa_kind && (!L->ki_codes_pool || !L->ki_scales_pool || !L->qi_codes || !L->qi_scales ||
                   !L->topk_idx || !L->topk_cnt || (L->ring_xi && !L->xi_new)))
    return CSA_ERR_INVALID_ARG;
  if (!al16(L->k_pool) || !al16(L->v_pool) || !al16(L->ring_k) || !al16(L->ring_v) ||
      !al16(L->k_new) || !al16(L->v_new) || !al16(L->q) || !al16(L->out) ||
      !al16(L->block_table) || (uintptr_t)L->ring_logits % 4 || (uintptr_t)L->logit_new % 4 ||
      (L->lse && (uintptr_t)L->lse % 4))
    return CSA_ERR_ALIGN;
  if (csa_kind && (!al16(L->ki_codes_pool) || !al16(L->ki_scales_pool) || !al16(L->qi_codes) ||
                   !al16(L->topk_idx) || !al4(L->topk_cnt) ||
                   (L->ring_xi && (!al16(L->ring_xi) || !al16(L->xi_new)))))
    return CSA_ERR_ALIGN;
  if (L->B < 1 || L->H < 1 || L->N < 0 || L->W < 0 || L->n_pages < 1 || L->max_blocks < 1)
    return CSA_ERR_INVALID_ARG;
  if ((L->N + 1 + kPageTokens - 1) / kPageTokens > L->max_blocks) return CSA_ERR_SHAPE;
  if (L->d != 128 || L->W > 128 || !pow2(L->m)) return CSA_ERR_UNSUPPORTED;
  if (csa_kind && (L->m > 32 || L->d_I != 64 || !(L->H_I == 1 || L->H_I == 2 || L->H_I == 4) ||
                   L->k < 1))
    return CSA_ERR_UNSUPPORTED;
  if (!csa_kind && L->m > 128) return CSA_ERR_UNSUPPORTED;
  if ((int64_t)L->B * L->max_blocks > ((int64_t)1 << 31)) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}
}  // namespace

extern "C" {

size_t csa_paged_decode_workspace_size(const csa_paged_layer* layer) {
  return check_paged(layer) == CSA_OK ? paged_ws(layer) : 0;
}

static csa_status paged_step(const csa_paged_layer* L, void* ws, cudaStream_t st);

csa_status csa_paged_decode_step(const csa_paged_layer* L, void* ws, size_t ws_bytes,
                                 void* stream) {
  csa_status s = check_paged(L);
  if (s != CSA_OK) return s;
  const size_t need = paged_ws(L);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !al16(ws))) return CSA_ERR_WORKSPACE;
  return paged_step(L, ws, static_cast<cudaStream_t>(stream));
}

size_t csa_paged_layer_pair_workspace_size(const csa_paged_layer* csa,
                                           const csa_paged_layer* hca) {
  return round_up(csa_paged_decode_workspace_size(csa), 256) +
         csa_paged_decode_workspace_size(hca);
}

csa_status csa_paged_layer_pair(const csa_paged_layer* csa, const csa_paged_layer* hca, void* ws,
                                size_t ws_bytes, void* stream) {
  if (!csa || !hca || csa->kind != 0 || hca->kind != 1) return CSA_ERR_INVALID_ARG;
  csa_status s = check_paged(csa);
  if (s != CSA_OK) return s;
  if ((s = check_paged(hca)) != CSA_OK) return s;
  const size_t need = csa_paged_layer_pair_workspace_size(csa, hca);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !al16(ws))) return CSA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the HCA layer on the library's side stream beside the CSA layer, as in csa_hca_layer_pair
  SideStreams* ss = side_streams(st);
  if (ss && (cudaEventRecord(ss->ev[0], st) != cudaSuccess ||
             cudaStreamWaitEvent(ss->s[0], ss->ev[0], 0) != cudaSuccess))
    return CSA_ERR_CUDA;
  uint8_t* ws_c = static_cast<uint8_t*>(ws);
  uint8_t* ws_h = ws_c + round_up(paged_ws(csa), 256);
  if ((s = paged_step(csa, ws_c, st)) != CSA_OK) return s;
  if ((s = paged_step(hca, ws_h, ss ? ss->s[0] : st)) != CSA_OK) return s;
  if (ss && (cudaEventRecord(ss->ev[2], ss->s[0]) != cudaSuccess ||
             cudaStreamWaitEvent(st, ss->ev[2], 0) != cudaSuccess))
    return CSA_ERR_CUDA;
  return CSA_OK;
}

// One validated paged decode step on stream st.
static csa_status paged_step(const csa_paged_layer* L, void* ws, cudaStream_t st) {
  csa_status s = CSA_OK;
  uint32_t* status = status_word();
  if (!status) return CSA_ERR_CUDA;
  const bool csa_kind = L->kind == 0;
  PagedLayout P;
  P.d = L->d;
  P.m = L->m;
  P.d_I = csa_kind ? L->d_I : 0;
  P.k_pool = L->k_pool;
  P.v_pool = L->v_pool;
  P.ki_codes_pool = csa_kind ? L->ki_codes_pool : nullptr;
  P.ki_scales_pool = csa_kind ? L->ki_scales_pool : nullptr;
  P.block_table = L->block_table;
  P.n_pages = L->n_pages;
  P.max_blocks = L->max_blocks;
  P.ring_k = L->ring_k;
  P.ring_v = L->ring_v;
  P.ring_logits = L->ring_logits;
  P.ring_xi = csa_kind ? L->ring_xi : nullptr;
  const int64_t t = L->N;  // the appended token's position
  if (launch_paged_append(P, L->B, L->k_new, L->v_new, L->logit_new,
                          csa_kind ? L->xi_new : nullptr, t, status, st) != cudaSuccess)
    return CSA_ERR_CUDA;
  const int64_t E = (t + 1) / L->m;  // entries visible to the new token
  AttendArgs a{L->q, L->k_pool, L->v_pool, nullptr, nullptr, L->ring_k, L->ring_v, L->out, L->lse,
               E, t + 1, t, 0, L->m, L->W, L->B, 1, L->H, L->d};
  a.paged = &P;
  if (csa_kind) {
    uint16_t* sc = static_cast<uint16_t*>(ws);
    // The append launched just above is the only kernel this one may overlap: it writes the
    // index key of the block the token closes (entry E - 1) and nothing else the indexer reads.
    Freshness fr;
    fr.keys_from = (t + 1) % L->m == 0 ? E - 1 : E;
    fr.queries = false;
    s = run_indexer(L->qi_codes, L->qi_scales, L->ki_codes_pool, L->ki_scales_pool, L->B, 1, t, E,
                    L->m, L->H_I, L->d_I, sc, nullptr, st, &P, fr);
    if (s != CSA_OK) return s;
    if (launch_topk(sc, L->B, 1, t, E, L->m, L->k, L->topk_idx, L->topk_cnt, st, true) !=
        cudaSuccess)
      return CSA_ERR_CUDA;
    a.topk_idx = L->topk_idx;
    a.topk_cnt = L->topk_cnt;
    a.k = L->k;
    return from_cuda(launch_attend(a, (int64_t)L->k + L->W, ws, status, st));
  }
  return from_cuda(launch_attend(a, E + L->W, ws, status, st));
}


size_t csa_shard_candidates_workspace_size(int B, int64_t E, int k) {
  (void)k;
  if (B < 1 || E < 0) return 0;
  return round_up((size_t)B * (size_t)E * 2, 256);
}

csa_status csa_shard_candidates(const uint8_t* qi_codes, const uint8_t* qi_scales,
                                const uint8_t* ki_codes, const uint8_t* ki_scales, int B,
                                int64_t q_pos0, int64_t E, int m, int H_I, int d_I, int k,
                                int32_t* cand_idx, uint16_t* cand_scores, int32_t* cand_cnt,
                                void* ws, size_t ws_bytes, void* stream) {
  csa_status s = check_index(qi_codes, qi_scales, ki_codes, ki_scales, B, 1, q_pos0, E, m, H_I,
                             d_I, k, cand_idx, cand_cnt, nullptr);
  if (s != CSA_OK) return s;
  if (!cand_scores) return CSA_ERR_INVALID_ARG;
  if (!al16(cand_scores)) return CSA_ERR_ALIGN;
  const size_t need = csa_shard_candidates_workspace_size(B, E, k);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !al16(ws))) return CSA_ERR_WORKSPACE;
  uint32_t* status = status_word();
  if (!status) return CSA_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* sc = static_cast<uint16_t*>(ws);  // the shard's BF16 scores
  s = run_index_topk(qi_codes, qi_scales, ki_codes, ki_scales, B, 1, q_pos0, E, m, H_I, d_I, k,
                     cand_idx, cand_cnt, sc, nullptr, st);
  if (s != CSA_OK) return s;
  return from_cuda(launch_candidates(sc, B, E, cand_idx, cand_cnt, k, cand_scores, status, st));
}

csa_status csa_topk_merge(const uint16_t* cand_scores, const int32_t* cand_idx,
                          const int32_t* cand_cnt, const int64_t* shard_base, int B, int S, int k,
                          int32_t* topk_idx, int32_t* topk_cnt, int32_t* shard_idx,
                          int32_t* shard_cnt, void* stream) {
  if (!cand_scores || !cand_idx || !cand_cnt || !shard_base || !topk_idx || !topk_cnt ||
      !shard_idx || !shard_cnt)
    return CSA_ERR_INVALID_ARG;
  if (!al16(cand_scores) || !al16(cand_idx) || !al16(topk_idx) || !al16(shard_idx))
    return CSA_ERR_ALIGN;
  if (B < 1 || S < 1 || k < 1) return CSA_ERR_INVALID_ARG;
  if (S > kMaxShards || k > 2048) return CSA_ERR_UNSUPPORTED;
  for (int i = 0; i < S; ++i)
    if (shard_base[i] < 0 || (i > 0 && shard_base[i] < shard_base[i - 1]) ||
        shard_base[i] + k > ((int64_t)1 << 31))
      return CSA_ERR_SHAPE;
  return from_cuda(launch_topk_merge(cand_scores, cand_idx, cand_cnt, shard_base, B, S, k, topk_idx,
                                     topk_cnt, shard_idx, shard_cnt,
                                     static_cast<cudaStream_t>(stream)));
}

csa_status csa_lse_merge(const uint16_t* parts, const float* parts_lse, int S, int64_t rows, int d,
                         uint16_t* out, float* lse, void* stream) {
  if (!parts || !parts_lse || !out) return CSA_ERR_INVALID_ARG;
  if (!al16(parts) || !al16(out) || (uintptr_t)parts_lse % 4 || (lse && (uintptr_t)lse % 4))
    return CSA_ERR_ALIGN;
  if (S < 1 || rows < 0) return CSA_ERR_INVALID_ARG;
  if (d % 8 != 0 || d < 8 || d > 1024) return CSA_ERR_UNSUPPORTED;
  if (rows == 0) return CSA_OK;
  return from_cuda(launch_lse_merge(parts, parts_lse, S, rows, d, out, lse,
                                    static_cast<cudaStream_t>(stream)));
}

csa_status csa_scatter_rows(const csa_copy_desc* descs, int n, void* stream) {
  if (n < 0 || n > CSA_MAX_COPIES || (n > 0 && !descs)) return CSA_ERR_INVALID_ARG;
  static_assert(CSA_MAX_COPIES == kMaxScatterCopies, "copy limits agree");
  ScatterCopy c[kMaxScatterCopies];
  int m = 0;
  for (int i = 0; i < n; ++i) {
    const csa_copy_desc& d = descs[i];
    if (d.rows < 0 || d.row_bytes < 0 || (d.rows > 1 && d.dst_stride < d.row_bytes))
      return CSA_ERR_INVALID_ARG;
    if (d.rows == 0 || d.row_bytes == 0) continue;
    if (!d.dst || !d.src) return CSA_ERR_INVALID_ARG;
    c[m++] = ScatterCopy{d.dst, d.src, d.rows, d.row_bytes, d.dst_stride};
  }
  return from_cuda(launch_scatter_rows(c, m, static_cast<cudaStream_t>(stream)));
}

int csa_abi_version(void) { return 3; }

csa_status csa_test_set_faults(long long wait_budget_cycles, uint32_t skip_mask) {
  if (skip_mask & ~CSA_FAULT_ALL) return CSA_ERR_INVALID_ARG;
  g_wait_budget.store(wait_budget_cycles > 0 ? wait_budget_cycles : 0);
  g_fault_mask.store(skip_mask);
  return CSA_OK;
}

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_SHAPE: return "inconsistent shape";
    case CSA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_DEVICE: return "device-side fault recorded";
  }
  return "unknown status";
}

csa_status csa_compress(const uint16_t* k_raw, const uint16_t* v_raw, const float* logits, int B,
                        int64_t N, int d, int m, int64_t tok_begin, int64_t tok_end,
                        uint16_t* k_cmp, uint16_t* v_cmp, void* stream) {
  csa_status s = check_compress(k_raw, v_raw, logits, B, N, d, m, tok_begin, tok_end, k_cmp, v_cmp);
  if (s != CSA_OK) return s;
  const int64_t j0 = tok_begin / m, j1 = tok_end / m;
  return from_cuda(launch_compress(k_raw, v_raw, logits, B, N, d, m, j0, j1 - j0, k_cmp, v_cmp,
                                   static_cast<cudaStream_t>(stream)));
}

csa_status csa_compress_index_keys(const uint16_t* xi_raw, const float* logits, int B, int64_t N,
                                   int d_I, int m, int64_t tok_begin, int64_t tok_end,
                                   uint8_t* ki_codes, uint8_t* ki_scales, void* stream) {
  csa_status s = check_index_keys(xi_raw, logits, B, N, d_I, m, tok_begin, tok_end, ki_codes,
                                  ki_scales);
  if (s != CSA_OK) return s;
  const int64_t j0 = tok_begin / m, j1 = tok_end / m;
  return from_cuda(launch_index_keys(xi_raw, logits, B, N, d_I, m, j0, j1 - j0, ki_codes,
                                     ki_scales, static_cast<cudaStream_t>(stream)));
}

csa_status csa_quantize_mxfp4(const uint16_t* x, int64_t rows, int d, uint8_t* codes,
                              uint8_t* scales, void* stream) {
  if (!x || !codes || !scales) return CSA_ERR_INVALID_ARG;
  if (!al16(x) || !al16(codes)) return CSA_ERR_ALIGN;
  if (rows < 0) return CSA_ERR_SHAPE;
  if (d != 32 && d != 64 && d != 128) return CSA_ERR_UNSUPPORTED;
  return from_cuda(launch_mxfp4_quantize(x, rows, d, codes, scales,
                                         static_cast<cudaStream_t>(stream)));
}

size_t csa_index_topk_workspace_size(int B, int Nq, int64_t E, int k, int scores_given) {
  (void)k;
  if (B < 1 || Nq < 1 || E < 0) return 0;
  return index_ws_bytes(B, Nq, E, scores_given);
}

csa_status csa_index_topk(const uint8_t* qi_codes, const uint8_t* qi_scales,
                          const uint8_t* ki_codes, const uint8_t* ki_scales, int B, int Nq,
                          int64_t q_pos0, int64_t E, int m, int H_I, int d_I, int k,
                          int32_t* topk_idx, int32_t* topk_cnt, uint16_t* scores, void* ws,
                          size_t ws_bytes, void* stream) {
  csa_status s = check_index(qi_codes, qi_scales, ki_codes, ki_scales, B, Nq, q_pos0, E, m, H_I,
                             d_I, k, topk_idx, topk_cnt, scores);
  if (s != CSA_OK) return s;
  const size_t need = index_ws_bytes(B, Nq, E, scores != nullptr);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !al16(ws))) return CSA_ERR_WORKSPACE;
  return run_index_topk(qi_codes, qi_scales, ki_codes, ki_scales, B, Nq, q_pos0, E, m, H_I, d_I,
                        k, topk_idx, topk_cnt, scores, ws, static_cast<cudaStream_t>(stream));
}

size_t csa_topk_workspace_size(int B, int Nq, int64_t E, int k) {
  (void)B; (void)Nq; (void)E; (void)k;
  return 0;
}

csa_status csa_index_scores(const uint8_t* qi_codes, const uint8_t* qi_scales,
                            const uint8_t* ki_codes, const uint8_t* ki_scales, int B, int Nq,
                            int64_t q_pos0, int64_t E, int m, int H_I, int d_I, uint16_t* scores,
                            float* scores_f32, void* stream) {
  if (!scores) return CSA_ERR_INVALID_ARG;
  if (scores_f32 && !al16(scores_f32)) return CSA_ERR_ALIGN;
  csa_status s = check_index_inputs(qi_codes, qi_scales, ki_codes, ki_scales, B, Nq, q_pos0, E,
                                    m, H_I, d_I, scores);
  if (s != CSA_OK) return s;
  return run_indexer(qi_codes, qi_scales, ki_codes, ki_scales, B, Nq, q_pos0, E, m, H_I, d_I,
                     scores, scores_f32, static_cast<cudaStream_t>(stream));
}

csa_status csa_topk_f32(const float* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                        int k, int32_t* topk_idx, int32_t* topk_cnt, void* stream) {
  csa_status s = check_topk(reinterpret_cast<const uint16_t*>(scores), B, Nq, q_pos0, E, m, k,
                            topk_idx, topk_cnt);
  if (s != CSA_OK) return s;
  const int64_t n_max = std::min(E, (q_pos0 + Nq) / m);
  if (n_max > 16 * 32768) return CSA_ERR_UNSUPPORTED;
  return from_cuda(launch_topk_f32(scores, B, Nq, q_pos0, E, m, k, topk_idx, topk_cnt,
                                   static_cast<cudaStream_t>(stream)));
}

csa_status csa_topk(const uint16_t* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                    int k, int32_t* topk_idx, int32_t* topk_cnt, void* ws, size_t ws_bytes,
                    void* stream) {
  (void)ws; (void)ws_bytes;
  csa_status s = check_topk(scores, B, Nq, q_pos0, E, m, k, topk_idx, topk_cnt);
  if (s != CSA_OK) return s;
  return from_cuda(launch_topk(scores, B, Nq, q_pos0, E, m, k, topk_idx, topk_cnt,
                               static_cast<cudaStream_t>(stream)));
}

size_t csa_attend_workspace_size(int B, int Nq, int H, int d, int k, int W) {
  if (B < 1 || Nq < 1 || H < 1 || k < 0 || W < 0) return 0;
  return attend_workspace_bytes(B * Nq, H, d, (int64_t)k + W);
}

csa_status csa_attend(const uint16_t* q, const uint16_t* k_cmp, const uint16_t* v_cmp, int64_t E,
                      const int32_t* topk_idx, const int32_t* topk_cnt, int k,
                      const uint16_t* k_raw, const uint16_t* v_raw, int64_t N, int W, int B,
                      int Nq, int64_t q_pos0, int H, int d, uint16_t* out, float* lse, void* ws,
                      size_t ws_bytes, void* stream) {
  csa_status s = check_attend(q, k_cmp, v_cmp, E, k_raw, v_raw, N, W, B, Nq, q_pos0, H, d, out, lse);
  if (s != CSA_OK) return s;
  if (!topk_idx || !topk_cnt || k < 0) return CSA_ERR_INVALID_ARG;
  if (!al16(topk_idx) || !al4(topk_cnt)) return CSA_ERR_ALIGN;
  const size_t need = attend_workspace_bytes(B * Nq, H, d, (int64_t)k + W);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !al16(ws))) return CSA_ERR_WORKSPACE;
  uint32_t* status = status_word();
  if (!status) return CSA_ERR_CUDA;
  AttendArgs a{q, k_cmp, v_cmp, topk_idx, topk_cnt, k_raw, v_raw, out, lse,
               E, N, q_pos0, k, 1, W, B, Nq, H, d};
  return from_cuda(launch_attend(a, (int64_t)k + W, ws, status, static_cast<cudaStream_t>(stream)));
}

size_t hca_attend_workspace_size(int B, int Nq, int H, int d, int64_t E, int m, int W) {
  if (B < 1 || Nq < 1 || H < 1 || E < 0 || m < 1 || W < 0) return 0;
  return attend_workspace_bytes(B * Nq, H, d, E + W);
}

csa_status hca_attend(const uint16_t* q, const uint16_t* k_cmp, const uint16_t* v_cmp, int64_t E,
                      int m, const uint16_t* k_raw, const uint16_t* v_raw, int64_t N, int W, int B,
                      int Nq, int64_t q_pos0, int H, int d, uint16_t* out, float* lse, void* ws,
                      size_t ws_bytes, void* stream) {
  csa_status s = check_attend(q, k_cmp, v_cmp, E, k_raw, v_raw, N, W, B, Nq, q_pos0, H, d, out, lse);
  if (s != CSA_OK) return s;
  if (m < 1) return CSA_ERR_INVALID_ARG;
  const size_t need = attend_workspace_bytes(B * Nq, H, d, E + W);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !al16(ws))) return CSA_ERR_WORKSPACE;
  uint32_t* status = status_word();
  if (!status) return CSA_ERR_CUDA;
  AttendArgs a{q, k_cmp, v_cmp, nullptr, nullptr, k_raw, v_raw, out, lse,
               E, N, q_pos0, 0, m, W, B, Nq, H, d};
  return from_cuda(launch_attend(a, E + W, ws, status, static_cast<cudaStream_t>(stream)));
}

size_t csa_hca_layer_pair_workspace_size(const csa_layer_desc* c, const hca_layer_desc* h) {
  // [CSA region: scores, then the CSA attention's partials][HCA region]: the two layers may run
  // concurrently, so their regions never overlap.
  return pair_csa_ws(c) + pair_hca_ws(h);
}

csa_status csa_hca_layer_pair(const csa_layer_desc* c, const hca_layer_desc* h, void* ws,
                              size_t ws_bytes, void* stream) {
  if (!c && !h) return CSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // validate everything before launching anything
  if (c) {
    if (c->m < 1) return CSA_ERR_INVALID_ARG;
    const int64_t E = c->N / c->m;
    csa_status s = check_compress(c->k_raw, c->v_raw, c->logits, c->B, c->N, c->d, c->m,
                                  c->compress_begin, c->N, c->k_cmp, c->v_cmp);
    if (s != CSA_OK) return s;
    s = check_index(c->qi_codes, c->qi_scales, c->ki_codes, c->ki_scales, c->B, c->Nq, c->q_pos0,
                    E, c->m, c->H_I, c->d_I, c->k, c->topk_idx, c->topk_cnt, c->scores);
    if (s != CSA_OK) return s;
    if (c->xi_raw) {
      s = check_index_keys(c->xi_raw, c->logits, c->B, c->N, c->d_I, c->m, c->compress_begin,
                           c->N, c->ki_codes, c->ki_scales);
      if (s != CSA_OK) return s;
    }
    s = check_attend(c->q, c->k_cmp, c->v_cmp, E, c->k_raw, c->v_raw, c->N, c->W, c->B, c->Nq,
                     c->q_pos0, c->H, c->d, c->out, c->lse);
    if (s != CSA_OK) return s;
  }
  if (h) {
    if (h->m < 1) return CSA_ERR_INVALID_ARG;
    const int64_t E = h->N / h->m;
    csa_status s = check_compress(h->k_raw, h->v_raw, h->logits, h->B, h->N, h->d, h->m,
                                  h->compress_begin, h->N, h->k_cmp, h->v_cmp);
    if (s != CSA_OK) return s;
    s = check_attend(h->q, h->k_cmp, h->v_cmp, E, h->k_raw, h->v_raw, h->N, h->W, h->B, h->Nq,
                     h->q_pos0, h->H, h->d, h->out, h->lse);
    if (s != CSA_OK) return s;
  }
  const size_t need = csa_hca_layer_pair_workspace_size(c, h);
  if (need > 0 && (ws == nullptr || ws_bytes < need || !al16(ws))) return CSA_ERR_WORKSPACE;
  uint32_t* status = status_word();
  if (!status) return CSA_ERR_CUDA;

  // Fork: with both layers present the HCA layer runs on a side stream beside the CSA layer
  // (a fork costs more than it saves for a single layer).
  SideStreams* ss = (c && h) ? side_streams(st) : nullptr;
  if (ss) {
    if (cudaEventRecord(ss->ev[0], st) != cudaSuccess ||
        cudaStreamWaitEvent(ss->s[0], ss->ev[0], 0) != cudaSuccess)
      return CSA_ERR_CUDA;
  }
  uint8_t* ws_c = static_cast<uint8_t*>(ws);
  uint8_t* ws_h = ws_c + pair_csa_ws(c);
  bool fused = false;  // the CSA decode layer ran as one launch (decode.cu)
  bool pool_late = false;  // the CSA layer's closed blocks are pooled with its scoring or after it
  if (c) {
    const int64_t E = c->N / c->m;
    const int64_t j0 = c->compress_begin / c->m;
    // Decode with 64 heads of dim 128 or fewer: indexer, top-k and attention in one launch,
    // which also pools the few blocks the step closes when no index keys are pooled with them.
    DecodePlan pl{};
    if (decode_indexer_fits(c->Nq, c->H_I, c->d_I) && c->d == 128 && c->H <= 64) {
      const int64_t nv = std::max<int64_t>(0, std::min<int64_t>(E, (c->q_pos0 + 1) / c->m));
      pl = plan_decode(c->B, E, nv, c->k, c->W, true, c->scores != nullptr);
    }
    const bool pool_inside = pl.ok && !c->xi_raw && E - j0 <= kDecodePoolMax;
    // Without the one-launch step, a decode-shaped layer may still pool the closed blocks in its
    // scoring launch (below); other shapes pool first, in a launch of their own.
    pool_late = !pl.ok && !c->xi_raw && E > j0 && E - j0 <= kDecodePoolMax &&
                decode_indexer_fits(c->Nq, c->H_I, c->d_I);
    if (!pool_inside && !pool_late &&
        launch_compress(c->k_raw, c->v_raw, c->logits, c->B, c->N, c->d, c->m, j0, E - j0,
                        c->k_cmp, c->v_cmp, st) != cudaSuccess)
      return CSA_ERR_CUDA;
    if (c->xi_raw &&
        launch_index_keys(c->xi_raw, c->logits, c->B, c->N, c->d_I, c->m, j0, E - j0,
                          const_cast<uint8_t*>(c->ki_codes), const_cast<uint8_t*>(c->ki_scales),
                          st) != cudaSuccess)
      return CSA_ERR_CUDA;
    if (pl.ok) {
      DecodeArgs a{};
      a.qi_codes = c->qi_codes;
      a.qi_scales = c->qi_scales;
      a.ki_codes = c->ki_codes;
      a.ki_scales = c->ki_scales;
      a.scores = c->scores;
      a.topk_idx = c->topk_idx;
      a.topk_cnt = c->topk_cnt;
      a.E = E;
      a.t = c->q_pos0;
      a.m = c->m;
      a.k = c->k;
      a.H_I = c->H_I;
      a.B = c->B;
      // When this call launched the pooling, the kernel's predecessor is known: the pooling of
      // the index keys from j0 on (xi_raw), else the entry pooling, which writes nothing the
      // indexer reads and the entries from j0 on. Otherwise the predecessor is unknown and the
      // kernel waits for it before reading anything.
      a.wait_first = pool_inside || E <= j0;
      a.keys_fresh_from = c->xi_raw ? j0 : E;
      a.attend = true;
      a.H = c->H;
      a.W = c->W;
      a.q = c->q;
      a.k_cmp = c->k_cmp;
      a.v_cmp = c->v_cmp;
      a.k_raw = c->k_raw;
      a.v_raw = c->v_raw;
      a.out = c->out;
      a.lse = c->lse;
      a.N = c->N;
      a.logits = c->logits;
      a.pool_j0 = pool_inside ? j0 : E;
      a.pool_j1 = E;
      if (launch_decode(a, pl, status, st) != cudaSuccess) return CSA_ERR_CUDA;
      fused = true;
    }
  }
  if (c && !fused) {
    const int64_t E = c->N / c->m;
    const int64_t j0 = c->compress_begin / c->m;
    Freshness fr;
    PoolRange pr{c->k_raw, c->v_raw, c->logits, c->k_cmp, c->v_cmp, c->N, j0, E};
    bool pooled = false;
    if (pool_late) {
      // no launch of this call precedes the scoring: it waits for its predecessor first
      fr.pool = &pr;
      fr.pooled = &pooled;
    } else if (E > j0) {
      fr.keys_from = c->xi_raw ? j0 : E;
      fr.queries = false;
    }
    csa_status s = run_index_topk(c->qi_codes, c->qi_scales, c->ki_codes, c->ki_scales, c->B,
                                  c->Nq, c->q_pos0, E, c->m, c->H_I, c->d_I, c->k, c->topk_idx,
                                  c->topk_cnt, c->scores, ws_c, st, fr);
    if (s != CSA_OK) return s;
    // the selection did not pool them: pool now, before the attention reads the entries
    if (pool_late && !pooled &&
        launch_compress(c->k_raw, c->v_raw, c->logits, c->B, c->N, c->d, c->m, j0, E - j0,
                        c->k_cmp, c->v_cmp, st) != cudaSuccess)
      return CSA_ERR_CUDA;
    AttendArgs a{c->q, c->k_cmp, c->v_cmp, c->topk_idx, c->topk_cnt, c->k_raw, c->v_raw, c->out,
                 c->lse, E, c->N, c->q_pos0, c->k, c->m, c->W, c->B, c->Nq, c->H, c->d};
    if (launch_attend(a, (int64_t)c->k + c->W, ws_c, status, st) != cudaSuccess) return CSA_ERR_CUDA;
  }
  if (h) {
    const int64_t E = h->N / h->m;
    const int64_t j0 = h->compress_begin / h->m;
    cudaStream_t sh = ss ? ss->s[0] : st;
    if (launch_compress(h->k_raw, h->v_raw, h->logits, h->B, h->N, h->d, h->m, j0, E - j0,
                        h->k_cmp, h->v_cmp, sh) != cudaSuccess)
      return CSA_ERR_CUDA;
    AttendArgs a{h->q, h->k_cmp, h->v_cmp, nullptr, nullptr, h->k_raw, h->v_raw, h->out, h->lse,
                 E, h->N, h->q_pos0, 0, h->m, h->W, h->B, h->Nq, h->H, h->d};
    // The compress launch just above is the attention's predecessor; it waits for its own
    // predecessor before letting the attention start, so the entries below j0 are complete.
    a.fresh_from = j0;
    if (launch_attend(a, hca_max_keys(E, h->m, h->N, h->W), ws_h, status, sh) != cudaSuccess)
      return CSA_ERR_CUDA;
  }
  if (ss) {  // join: the caller's stream continues after both side streams
    if (cudaEventRecord(ss->ev[2], ss->s[0]) != cudaSuccess ||
        cudaStreamWaitEvent(st, ss->ev[2], 0) != cudaSuccess)
      return CSA_ERR_CUDA;
  }
  return CSA_OK;
}

csa_status csa_get_device_status(void* stream, int reset, uint32_t* flags_out) {
  uint32_t* status = status_word();
  if (!status) return CSA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  if (reset && cudaMemset(status, 0, sizeof(uint32_t)) != cudaSuccess) return CSA_ERR_CUDA;
  if (flags_out) *flags_out = v;
  return v ? CSA_ERR_DEVICE : CSA_OK;
}

}  // extern "C"
