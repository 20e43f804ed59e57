// Per-query top-k over BF16 index scores (9fzt.com DeepSeek-V4 summary, item 4: the selector
// runs on BF16 scores; Lighthouse "deep deepseek v4 release" 八.3: top-k over compressed
// entries). Order: score descending, ties to the lower entry index; output sorted ascending,
// padded with -1; count = min(k, visible).
//
// One CTA per query row. BF16 scores map to order-preserving 16-bit keys, so selection is an
// exact two-digit radix select (high byte, then low byte) followed by an ordered compaction:
// everything above the threshold key T, plus the lowest-index entries equal to T until k are
// taken. The row is cached in shared memory when it fits; otherwise it is re-read from L2.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kTopkThreads = 512;
constexpr int kSmemKeys = 48 * 1024;  // keys cached in shared memory (96 KB)

CSA_DEV uint32_t order_key(uint32_t bits) {
  if (bits == 0x8000u) bits = 0u;  // -0 counts as +0
  return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
}

// Finds the bin b with count(bins > b) < need <= count(bins >= b) over 256 bins; returns the bin
// and count(bins > b). Called by all threads; uses warp 0.
CSA_DEV void select_bin(const uint32_t* hist, uint32_t need, int* out_bin, uint32_t* out_above) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    // lane owns bins [248 - 8*lane .. 255 - 8*lane] (descending blocks of 8)
    uint32_t local[8];
    uint32_t tot = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      local[q] = hist[255 - (lane * 8 + q)];
      tot += local[q];
    }
    // inclusive scan over lanes (descending bin order)
    uint32_t inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const uint32_t exc = inc - tot;
    if (exc < need && need <= inc) {
      uint32_t run = exc;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (run < need && need <= run + local[q]) {
          *out_bin = 255 - (lane * 8 + q);
          *out_above = run;
        }
        run += local[q];
      }
    }
  }
}

// Block-wide exclusive scan of two counters (one per thread).
CSA_DEV void block_exclusive_scan2(uint32_t a, uint32_t b, uint32_t* ex_a, uint32_t* ex_b,
                                   uint32_t* warp_a, uint32_t* warp_b) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t va = __shfl_up_sync(0xffffffffu, ia, o);
    uint32_t vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += va;
      ib += vb;
    }
  }
  if (lane == 31) {
    warp_a[w] = ia;
    warp_b[w] = ib;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    uint32_t xa = lane < nw ? warp_a[lane] : 0u, xb = lane < nw ? warp_b[lane] : 0u;
    uint32_t sa = xa, sb = xb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t va = __shfl_up_sync(0xffffffffu, sa, o);
      uint32_t vb = __shfl_up_sync(0xffffffffu, sb, o);
      if (lane >= o) {
        sa += va;
        sb += vb;
      }
    }
    if (lane < nw) {
      warp_a[lane] = sa - xa;
      warp_b[lane] = sb - xb;
    }
  }
  __syncthreads();
  *ex_a = warp_a[w] + ia - a;
  *ex_b = warp_b[w] + ib - b;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const uint16_t* __restrict__ scores,
                                                            int Nq, int64_t q_pos0, int64_t E,
                                                            int m, int k, int64_t cap,
                                                            int32_t* __restrict__ topk_idx,
                                                            int32_t* __restrict__ topk_cnt) {
  extern __shared__ uint16_t skeys[];  // `cap` keys
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_a[32], warp_b[32];
  __shared__ int sh_bin;
  __shared__ uint32_t sh_above;

  const int64_t row = blockIdx.x;  // b * Nq + i
  const int64_t t = q_pos0 + (row % Nq);
  const int64_t n = max((int64_t)0, min(E, (t + 1) / m));
  const uint16_t* src = scores + row * E;
  int32_t* out = topk_idx + row * (int64_t)k;
  const int tid = threadIdx.x, nt = blockDim.x;

  if (n <= k) {
    for (int64_t r = tid; r < k; r += nt) out[r] = (r < n) ? (int32_t)r : -1;
    if (tid == 0) topk_cnt[row] = (int32_t)n;
    return;
  }
  const bool cached = n <= cap;
  if (cached) {
    for (int64_t r = tid; r < n; r += nt) skeys[r] = (uint16_t)order_key(src[r]);
  }
  auto key_at = [&](int64_t r) -> uint32_t {
    return cached ? (uint32_t)skeys[r] : order_key(src[r]);
  };

  // ---- digit 1: high byte ----
  for (int q = tid; q < 256; q += nt) hist[q] = 0u;
  __syncthreads();
  for (int64_t r = tid; r < n; r += nt) atomicAdd(&hist[key_at(r) >> 8], 1u);
  __syncthreads();
  select_bin(hist, (uint32_t)k, &sh_bin, &sh_above);
  __syncthreads();
  const uint32_t hi = (uint32_t)sh_bin;
  const uint32_t above_hi = sh_above;
  __syncthreads();
  // ---- digit 2: low byte within the high bin ----
  for (int q = tid; q < 256; q += nt) hist[q] = 0u;
  __syncthreads();
  for (int64_t r = tid; r < n; r += nt) {
    const uint32_t kk = key_at(r);
    if ((kk >> 8) == hi) atomicAdd(&hist[kk & 0xFFu], 1u);
  }
  __syncthreads();
  select_bin(hist, (uint32_t)k - above_hi, &sh_bin, &sh_above);
  __syncthreads();
  const uint32_t T = (hi << 8) | (uint32_t)sh_bin;
  const uint32_t n_gt = above_hi + sh_above;
  const uint32_t need_eq = (uint32_t)k - n_gt;

  // ---- ordered compaction over contiguous per-thread segments ----
  const int64_t seg = (n + nt - 1) / nt;
  const int64_t r0 = min(n, seg * tid), r1 = min(n, r0 + seg);
  uint32_t c_gt = 0, c_eq = 0;
  for (int64_t r = r0; r < r1; ++r) {
    const uint32_t kk = key_at(r);
    c_gt += kk > T;
    c_eq += kk == T;
  }
  uint32_t gt_before, eq_before;
  block_exclusive_scan2(c_gt, c_eq, &gt_before, &eq_before, warp_a, warp_b);
  for (int64_t r = r0; r < r1; ++r) {
    const uint32_t kk = key_at(r);
    if (kk > T) {
      out[gt_before + min(eq_before, need_eq)] = (int32_t)r;
      ++gt_before;
    } else if (kk == T) {
      if (eq_before < need_eq) out[gt_before + eq_before] = (int32_t)r;
      ++eq_before;
    }
  }
  if (tid == 0) topk_cnt[row] = k;
}

}  // namespace

cudaError_t launch_topk(const uint16_t* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                        int k, int32_t* topk_idx, int32_t* topk_cnt, cudaStream_t stream) {
  const int64_t rows = (int64_t)B * Nq;
  if (rows <= 0) return cudaSuccess;
  int64_t max_vis = min(E, (q_pos0 + Nq) / m);
  if (max_vis < 0) max_vis = 0;
  const int64_t cap = max_vis > k ? min(max_vis, (int64_t)kSmemKeys) : 0;
  const size_t smem = (size_t)cap * 2;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemKeys * 2);
  if (e != cudaSuccess) return e;
  ProfScope prof(stream, "topk");
  topk_kernel<<<(unsigned)rows, kTopkThreads, smem, stream>>>(scores, Nq, q_pos0, E, m, k, cap,
                                                              topk_idx, topk_cnt);
  return cudaGetLastError();
}

}  // namespace csa
