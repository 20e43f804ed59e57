// The exchange steps of an entry-sharded CSA decode: the entries of a sequence are split over S
// shards (GPUs, or slices of one GPU's cache), every shard selects its own top-k candidates, the
// candidates are merged into the global top-k, every shard attends to its share of the global
// selection, and the shards' partial attention outputs are merged by their log-sum-exp.
//
// Lighthouse "deep deepseek v4 release" 八.3: the top-k and the attention over the kept entries
// plus the window; the pages' 1M-token context (9fzt.com DeepSeek-V4 summary, item 1) is what
// makes a sequence's entries worth splitting. The global selection is exactly the unsharded one:
// every entry of the global top-k is among its own shard's top-k, so the merge sees it, and the
// order (score descending, ties to the lower global index) is decided on the same BF16 scores.
//
//   candidates_kernel  the BF16 scores of one shard's selected entries (its candidates)
//   topk_merge_kernel  one CTA per sequence: an exact radix select over the S x k candidates
//                      (shard-major layouts: candidates and per-shard lists [S, B, k])
//                      (17-bit keys: the order-preserving score key, and 0 for no candidate),
//                      then the ordered write of the global list and of each shard's part of it
//   lse_merge_kernel   out = sum_s e^(lse_s - L) out_s with L = log sum_s e^(lse_s)
#include "common.cuh"
#include "kernels.h"
#include "prof.h"
#include "select.cuh"

namespace csa {
namespace {

constexpr int kMergeThreads = 256;

// The BF16 score of every selected entry of one shard (0 past the count).
__global__ void candidates_kernel(const uint16_t* __restrict__ scores, int64_t E,
                                  const int32_t* __restrict__ sel, const int32_t* __restrict__ cnt,
                                  int k, uint16_t* __restrict__ cand_scores, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t b = blockIdx.y;
  const int c = cnt[b];
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < k; j += gridDim.x * blockDim.x) {
    const int32_t l = j < c ? sel[b * k + j] : -1;
    uint16_t v = 0;
    if (l >= 0 && l < E)
      v = scores[b * E + l];
    else if (l >= E)
      atomicOr(status, kFlagBadIndex);
    cand_scores[b * k + j] = v;
  }
}

struct ShardBases {
  int64_t base[kMaxShards];  // first global entry index of each shard
};

__global__ void __launch_bounds__(kMergeThreads) topk_merge_kernel(
    const uint16_t* __restrict__ cand_scores, const int32_t* __restrict__ cand_idx,
    const int32_t* __restrict__ cand_cnt, const ShardBases bases, int B, int S, int k,
    int32_t* __restrict__ topk_idx, int32_t* __restrict__ topk_cnt,
    int32_t* __restrict__ shard_idx, int32_t* __restrict__ shard_cnt) {
  extern __shared__ uint32_t mkey[];  // [S * k] 0 = no candidate, else order key + 1
  __shared__ uint32_t hist[257];
  __shared__ uint32_t wa[33], wb[33];
  __shared__ int sh_bin;
  __shared__ uint32_t sh_above;
  __shared__ uint32_t sh_first[kMaxShards];  // first output position of each shard's entries
  pdl_trigger();
  pdl_wait();
  const int64_t b = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = S * k;
  uint32_t valid_total = 0;
  for (int p = tid; p < n; p += kMergeThreads) {
    const int s = p / k, j = p % k;
    const int c = min(max(cand_cnt[s * B + b], 0), k);
    uint32_t key = 0;
    if (j < c && cand_idx[(s * B + b) * (int64_t)k + j] >= 0)
      key = order_key(cand_scores[(s * B + b) * (int64_t)k + j]) + 1u;
    mkey[p] = key;
    valid_total += key != 0u;
  }
  // the selection size: min(k, candidates)
  for (int o = 16; o > 0; o >>= 1) valid_total += __shfl_xor_sync(0xffffffffu, valid_total, o);
  for (int i = tid; i < 257; i += kMergeThreads) hist[i] = 0u;
  if (tid == 0) sh_above = 0u;
  __syncthreads();
  if ((tid & 31) == 0) atomicAdd(&sh_above, valid_total);
  __syncthreads();
  const uint32_t nvalid = sh_above;
  const uint32_t cnt = min((uint32_t)k, nvalid);
  __syncthreads();
  // exact threshold: digit 1 = key >> 8 (0 .. 256), digit 2 = key & 255 inside it
  uint32_t T = 0, need_eq = 0;
  if (cnt > 0) {
    for (int p = tid; p < n; p += kMergeThreads)
      if (mkey[p]) atomicAdd(&hist[mkey[p] >> 8], 1u);
    __syncthreads();
    if (tid == 0) {
      uint32_t run = 0;
      int bin = 256;
      for (; bin >= 0; --bin) {
        if (run + hist[bin] >= cnt) break;
        run += hist[bin];
      }
      sh_bin = bin;
      sh_above = run;
    }
    __syncthreads();
    const uint32_t hb = (uint32_t)sh_bin, above_hi = sh_above;
    __syncthreads();
    for (int i = tid; i < 257; i += kMergeThreads) hist[i] = 0u;
    __syncthreads();
    for (int p = tid; p < n; p += kMergeThreads)
      if (mkey[p] && (mkey[p] >> 8) == hb) atomicAdd(&hist[mkey[p] & 255u], 1u);
    __syncthreads();
    if (tid == 0) {
      uint32_t run = above_hi;
      int bin = 255;
      for (; bin >= 0; --bin) {
        if (run + hist[bin] >= cnt) break;
        run += hist[bin];
      }
      sh_bin = bin;
      sh_above = run;
    }
    __syncthreads();
    T = (hb << 8) | (uint32_t)sh_bin;
    need_eq = cnt - sh_above;
  }
  // ordered write: every thread a contiguous run of positions (positions ascend with the global
  // index: shards cover increasing index ranges, each shard's candidates are ascending)
  const int seg = (n + kMergeThreads - 1) / kMergeThreads;
  const int p0 = min(n, tid * seg), p1 = min(n, p0 + seg);
  uint32_t c_gt = 0, c_eq = 0;
  if (cnt > 0)
    for (int p = p0; p < p1; ++p) {
      c_gt += mkey[p] > T;
      c_eq += mkey[p] == T;
    }
  uint32_t gb, eb, tg, te;
  block_scan2(c_gt, c_eq, &gb, &eb, &tg, &te, wa, wb);
  if (tid < S) sh_first[tid] = 0xFFFFFFFFu;
  __syncthreads();
  // global position of each selected candidate; the first selected position of every shard
  for (int p = p0; p < p1 && cnt > 0; ++p) {
    const uint32_t key = mkey[p];
    int pos = -1;
    if (key > T) {
      pos = (int)(gb + min(eb, need_eq));
      ++gb;
    } else if (key == T) {
      if (eb < need_eq) pos = (int)(gb + eb);
      ++eb;
    }
    mkey[p] = pos >= 0 ? 0x80000000u | (uint32_t)pos : 0u;  // reused: the output position
    if (pos >= 0) atomicMin(&sh_first[p / k], (uint32_t)pos);
  }
  __syncthreads();
  for (int p = tid; p < k; p += kMergeThreads)
    if ((uint32_t)p >= cnt) topk_idx[b * k + p] = -1;
  for (int p = tid; p < n; p += kMergeThreads) {
    const int s = p / k, j = p % k;
    const uint32_t v = mkey[p];
    if (v & 0x80000000u) {
      const int pos = (int)(v & 0x7FFFFFFFu);
      const int32_t local = cand_idx[(s * B + b) * (int64_t)k + j];
      topk_idx[b * k + pos] = (int32_t)(bases.base[s] + local);
      shard_idx[(s * B + b) * (int64_t)k + (pos - (int)sh_first[s])] = local;
    }
  }
  // each shard's count, then its list padded with -1
  __syncthreads();
  if (tid < S) {
    uint32_t c = 0;
    const uint32_t f = sh_first[tid];
    if (f != 0xFFFFFFFFu) {
      uint32_t nxt = cnt;
      for (int s2 = tid + 1; s2 < S; ++s2)
        if (sh_first[s2] != 0xFFFFFFFFu) {
          nxt = sh_first[s2];
          break;
        }
      c = nxt - f;
    }
    wa[tid] = c;
    shard_cnt[tid * B + b] = (int32_t)c;
  }
  if (tid == 0) topk_cnt[b] = (int32_t)cnt;
  __syncthreads();
  for (int p = tid; p < n; p += kMergeThreads) {
    const int s = p / k, j = p % k;
    if ((uint32_t)j >= wa[s]) shard_idx[(s * B + b) * (int64_t)k + j] = -1;
  }
}

// rows x d outputs of S shards: weights e^(lse_s - L), L = log sum_s e^(lse_s); a shard with an
// empty key set has lse = -inf and weight 0.
__global__ void lse_merge_kernel(const uint16_t* __restrict__ parts, const float* __restrict__ lse,
                                 int S, int64_t rows, int d, uint16_t* __restrict__ out,
                                 float* __restrict__ lse_out) {
  pdl_trigger();
  pdl_wait();
  const int per_row = d / 8;
  const int64_t total = rows * per_row;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = x / per_row;
    const int c8 = (int)(x % per_row);
    float L = -INFINITY;
    for (int s = 0; s < S; ++s) L = fmaxf(L, lse[s * rows + r]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float wsum = 0.f;
    if (L != -INFINITY) {
      for (int s = 0; s < S; ++s) {
        const float ls = lse[s * rows + r];
        if (ls == -INFINITY) continue;
        const float w = expf(ls - L);
        wsum += w;
        const uint4 v = *reinterpret_cast<const uint4*>(parts + (s * rows + r) * d + c8 * 8);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[2 * e] += w * bf16_bits_to_f32(u[e] & 0xFFFFu);
          acc[2 * e + 1] += w * bf16_bits_to_f32(u[e] >> 16);
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint4 o;
    o.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    o.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    o.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(out + r * d + c8 * 8) = o;
    if (lse_out && c8 == 0) lse_out[r] = L == -INFINITY ? -INFINITY : L + logf(wsum);
  }
}

}  // namespace

cudaError_t launch_candidates(const uint16_t* scores, int B, int64_t E, const int32_t* sel,
                              const int32_t* cnt, int k, uint16_t* cand_scores, uint32_t* status,
                              cudaStream_t stream) {
  dim3 grid((unsigned)((k + 255) / 256), (unsigned)B);
  ProfScope prof(stream, "shard_candidates");
  return launch_ex(candidates_kernel, grid, dim3(256), 0, stream, 1, scores, E, sel, cnt, k,
                   cand_scores, status);
}

cudaError_t launch_topk_merge(const uint16_t* cand_scores, const int32_t* cand_idx,
                              const int32_t* cand_cnt, const int64_t* shard_base, int B, int S,
                              int k, int32_t* topk_idx, int32_t* topk_cnt, int32_t* shard_idx,
                              int32_t* shard_cnt, cudaStream_t stream) {
  if (S < 1 || S > kMaxShards) return cudaErrorInvalidValue;
  ShardBases bases{};
  for (int s = 0; s < S; ++s) bases.base[s] = shard_base[s];
  const size_t smem = (size_t)S * k * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_merge_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ProfScope prof(stream, "topk_merge");
  return launch_ex(topk_merge_kernel, dim3((unsigned)B), dim3(kMergeThreads), smem, stream, 1,
                   cand_scores, cand_idx, cand_cnt, bases, B, S, k, topk_idx, topk_cnt, shard_idx,
                   shard_cnt);
}

cudaError_t launch_lse_merge(const uint16_t* parts, const float* lse, int S, int64_t rows, int d,
                             uint16_t* out, float* lse_out, cudaStream_t stream) {
  const int64_t total = rows * (d / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)kNumSMs * 8) blocks = (int64_t)kNumSMs * 8;
  if (blocks < 1) blocks = 1;
  ProfScope prof(stream, "shard_lse_merge");
  return launch_ex(lse_merge_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 1, parts, lse,
                   S, rows, d, out, lse_out);
}

}  // namespace csa
