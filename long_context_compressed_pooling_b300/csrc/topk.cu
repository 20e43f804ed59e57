// Per-query top-k over BF16 index scores (9fzt.com DeepSeek-V4 summary, item 4: the selector
// runs on BF16 scores; Lighthouse "deep deepseek v4 release" 八.3: top-k over compressed
// entries). Order: score descending, ties to the lower entry index; output sorted ascending,
// padded with -1; count = min(k, visible).
//
// BF16 scores map to order-preserving 16-bit keys, so selection is an exact two-digit radix
// select (high byte, then low byte) followed by an ordered compaction: every key above the
// threshold T, plus the lowest-index keys equal to T until k are taken.
//
// One CTA or thread-block cluster per query row, holding the row in registers: CTA rank r of
// a cluster of C owns a contiguous chunk of NT x KPT keys, every thread KPT contiguous keys of
// it. The shape is picked per launch: rows of up to 32768 keys with enough rows to fill the GPU
// (prefill) take one CTA per row, the smallest shape that holds the row (128 threads x 8 keys
// up to 1024 x 32); few rows (decode) are spread over clusters
// of 256-1024-thread CTAs so that the grid covers the SMs (a 32768-key row: 8 CTAs of 4096
// keys; a 262144-key row at 1M context: 16 CTAs of 16384). The cluster exchanges only the CTA
// maxima, 256-bin histograms and selected-key counts through distributed shared memory after
// hardware cluster barriers; every CTA derives the same threshold and writes its selected
// indices at their final, ascending positions. Rows longer than 16 x 32768 keys stage their
// chunks in shared memory instead. No grid-wide synchronisation and no spin waits are involved.
//
// Fast threshold: scores sit on the BF16 grid, so most of a row's top k lie within 255 grid
// steps of the row maximum. One histogram of (max - key) over those 255 steps finds T in a
// single pass; only when fewer than k keys fall in that band does the exact two-digit radix
// select run.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"
#include "select.cuh"

namespace csa {
namespace {

constexpr int kClusterThreads = 256;   // threads per CTA of a multi-CTA (cluster) row
constexpr int kMaxChunkKeys = 16384;   // keys one cluster CTA stages in shared memory (32 KB)

template <int NW>
struct TopkShared {
  uint32_t whist[NW * 256];  // per-warp histograms (plain shared atomics, no cross-warp contention)
  uint32_t wmax[32];
  uint32_t cta_max;          // this CTA's largest key (read by the cluster)
  uint32_t hist1[256];
  uint32_t hist2[256];
  uint32_t gsum[256];
  uint32_t wa[33], wb[33];
  uint32_t cta_gt, cta_eq;  // this CTA's keys above / equal to the threshold (read by the cluster)
  int bin;
  uint32_t above;
};

// NT threads per CTA; the cluster (1 to 16 CTAs) works on one row.
template <int NT>
__global__ void __launch_bounds__(NT) topk_kernel(const uint16_t* __restrict__ scores, int Nq,
                                                  int64_t q_pos0, int64_t E, int m, int k, int cap,
                                                  int32_t* __restrict__ topk_idx,
                                                  int32_t* __restrict__ topk_cnt) {
  constexpr int NW = NT / 32;
  extern __shared__ uint16_t skeys[];  // `cap` keys: this CTA's chunk when it fits
  __shared__ TopkShared<NW> sh;
  pdl_trigger();
  pdl_wait();
  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int64_t row = blockIdx.y;  // b * Nq + i
  const int64_t t = q_pos0 + (row % Nq);
  const int64_t n = max((int64_t)0, min(E, (t + 1) / m));
  const uint16_t* src = scores + row * E;
  int32_t* out = topk_idx + row * (int64_t)k;
  const int tid = threadIdx.x, nt = NT;

  if (n <= k) {  // uniform over the cluster: every CTA of it works on this row
    for (int64_t r = (int64_t)rank * nt + tid; r < k; r += (int64_t)C * nt)
      out[r] = (r < n) ? (int32_t)r : -1;
    if (rank == 0 && tid == 0) topk_cnt[row] = (int32_t)n;
    return;
  }

  const int64_t L = (n + C - 1) / C;
  const int64_t lo = min(n, (int64_t)rank * L), hi = min(n, lo + L);
  const int len = (int)(hi - lo);
  const bool cached = len <= cap;
  if (cached) {
    for (int r0 = tid; r0 < len; r0 += 4 * nt) {  // four independent loads in flight per thread
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = r0 + u * nt < len ? (uint32_t)src[lo + r0 + u * nt] : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (r0 + u * nt < len) skeys[r0 + u * nt] = (uint16_t)order_key(v[u]);
    }
  }
  auto key_at = [&](int r) -> uint32_t {
    return cached ? (uint32_t)skeys[r] : order_key(src[lo + r]);
  };
  uint32_t* wh = sh.whist + (tid >> 5) * 256;
  for (int q = tid; q < NW * 256; q += nt) sh.whist[q] = 0u;
  __syncthreads();

  // ---- the row's largest key -------------------------------------------------------------------
  uint32_t mx = 0;
  for (int r = tid; r < len; r += nt) mx = max(mx, key_at(r));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((tid & 31) == 0) sh.wmax[tid >> 5] = mx;
  __syncthreads();
  if (tid == 0) {
    uint32_t m2 = 0;
    for (int w = 0; w < NW; ++w) m2 = max(m2, sh.wmax[w]);
    sh.cta_max = m2;
  }
  __syncthreads();
  if (C > 1) cluster_sync();
  const uint32_t row_max = C > 1 ? cluster_max(&sh.cta_max, C) : sh.cta_max;

  // ---- near-max histogram: one bin per BF16 step below the maximum ---------------------------
  // The k-th largest key of a row with k << n sits a few octaves of BF16 steps below the
  // maximum, so only the keys within 255 steps are counted: few atomics and no hot bin (a
  // histogram of the high byte would pile almost every score into the same few bins).
  for (int r = tid; r < len; r += nt) {
    const uint32_t dd = row_max - key_at(r);
    if (dd < 255u) atomicAdd(&wh[dd], 1u);
  }
  __syncthreads();
  reduce_warp_hists<NW>(sh.whist, sh.hist1);
  __syncthreads();
  for (int q = tid; q < NW * 256; q += nt) sh.whist[q] = 0u;
  if (C > 1) {
    cluster_sync();
    for (int q = tid; q < 256; q += nt) sh.gsum[q] = cluster_sum(&sh.hist1[q], C);
  } else {
    for (int q = tid; q < 256; q += nt) sh.gsum[q] = sh.hist1[q];
  }
  __syncthreads();
  select_prefix(sh.gsum, (uint32_t)k, &sh.bin, &sh.above);
  __syncthreads();
  uint32_t T, need_eq;
  if (sh.bin >= 0) {
    T = row_max - (uint32_t)sh.bin;
    need_eq = (uint32_t)k - sh.above;
  } else {
    // Fallback (the k-th key lies further below the maximum): exact two-digit radix select.
    __syncthreads();
    // ---- digit 1: high byte ----
    for (int r = tid; r < len; r += nt) atomicAdd(&wh[key_at(r) >> 8], 1u);
    __syncthreads();
    reduce_warp_hists<NW>(sh.whist, sh.hist2);
    __syncthreads();  // every bin is summed before the per-warp histograms are cleared
    for (int q = tid; q < NW * 256; q += nt) sh.whist[q] = 0u;
    if (C > 1) {
      cluster_sync();
      for (int q = tid; q < 256; q += nt) sh.gsum[q] = cluster_sum(&sh.hist2[q], C);
    } else {
      for (int q = tid; q < 256; q += nt) sh.gsum[q] = sh.hist2[q];
    }
    __syncthreads();
    select_bin(sh.gsum, (uint32_t)k, &sh.bin, &sh.above);
    __syncthreads();
    const uint32_t hi_byte = (uint32_t)sh.bin;
    const uint32_t above_hi = sh.above;
    // ---- digit 2: low byte inside the high bin ----
    for (int r = tid; r < len; r += nt) {
      const uint32_t kk = key_at(r);
      if ((kk >> 8) == hi_byte) atomicAdd(&wh[kk & 0xFFu], 1u);
    }
    __syncthreads();
    reduce_warp_hists<NW>(sh.whist, sh.hist1);
    __syncthreads();
    if (C > 1) {
      cluster_sync();
      for (int q = tid; q < 256; q += nt) sh.gsum[q] = cluster_sum(&sh.hist1[q], C);
    } else {
      for (int q = tid; q < 256; q += nt) sh.gsum[q] = sh.hist1[q];
    }
    __syncthreads();
    select_bin(sh.gsum, (uint32_t)k - above_hi, &sh.bin, &sh.above);
    __syncthreads();
    T = (hi_byte << 8) | (uint32_t)sh.bin;
    need_eq = (uint32_t)k - (above_hi + sh.above);
  }

  // ---- ordered compaction: rounds of nt groups of 8 consecutive keys -------------------------
  const int groups = (len + 7) / 8;
  const int rounds = (groups + nt - 1) / nt;
  uint32_t my_gt = 0, my_eq = 0;
  for (int rd = 0; rd < rounds; ++rd) {
    const int g = rd * nt + tid;
    for (int j = 0; j < 8; ++j) {
      const int r = g * 8 + j;
      if (g < groups && r < len) {
        const uint32_t kk = key_at(r);
        my_gt += kk > T;
        my_eq += kk == T;
      }
    }
  }
  uint32_t ex_a, ex_b, cta_gt, cta_eq;
  block_scan2(my_gt, my_eq, &ex_a, &ex_b, &cta_gt, &cta_eq, sh.wa, sh.wb);
  if (tid == 0) {
    sh.cta_gt = cta_gt;
    sh.cta_eq = cta_eq;
  }
  __syncthreads();
  // keys of the lower-ranked CTAs of this row
  uint32_t gt_before = 0, eq_before = 0;
  if (C > 1) {
    cluster_sync();
    gt_before = cluster_sum(&sh.cta_gt, rank);
    eq_before = cluster_sum(&sh.cta_eq, rank);
  }
  for (int rd = 0; rd < rounds; ++rd) {
    const int g = rd * nt + tid;
    uint32_t c_gt = 0, c_eq = 0;
    uint32_t keys8[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = g * 8 + j;
      keys8[j] = (g < groups && r < len) ? key_at(r) : 0u;  // 0 is below every real key
      c_gt += keys8[j] > T;
      c_eq += keys8[j] == T;
    }
    uint32_t xg, xe, tg, te;
    block_scan2(c_gt, c_eq, &xg, &xe, &tg, &te, sh.wa, sh.wb);
    uint32_t gb = gt_before + xg, eb = eq_before + xe;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t kk = keys8[j];
      const int64_t idx = lo + (int64_t)g * 8 + j;
      // positions are < k by construction; the guard keeps any inconsistency inside the row
      if (kk > T) {
        const uint32_t pos = gb + min(eb, need_eq);
        if (pos < (uint32_t)k) out[pos] = (int32_t)idx;
        ++gb;
      } else if (kk == T) {
        if (eb < need_eq && gb + eb < (uint32_t)k) out[gb + eb] = (int32_t)idx;
        ++eb;
      }
    }
    gt_before += tg;
    eq_before += te;
  }
  if (rank == 0 && tid == 0) topk_cnt[row] = k;
  if (C > 1) cluster_sync();  // no CTA leaves while another may still read its shared memory
}


// Register-resident selection. A row is split over a cluster of C CTAs (C = 1 for rows that
// fit one CTA); CTA rank r owns the contiguous keys [r*NT*KPT, (r+1)*NT*KPT) and thread t of it
// the KPT keys starting at t*KPT inside that range, loaded with 16-byte loads when the row is
// 16-byte aligned. Max, near-max histogram, counts and the ordered write all run on registers;
// the cluster exchanges only its CTAs' maxima, histograms and counts through distributed shared
// memory (three hardware cluster barriers), and one block scan of per-thread selection masks
// orders the output because every thread's keys are contiguous and ranks follow key order.
//
// F32: FP32 scores with 32-bit keys. The threshold search runs on the upper 16 bits of the key
// first (the BF16-truncated score: near-max histogram, else the two-digit radix select), then
// resolves the keys in that bucket with two more byte digits of the lower half.
// NN: BF16 scores known to be non-negative with zero stored as +0 (the indexer's ReLU sums):
// their bit patterns already order like their values and serve as keys unchanged.
template <int NT, int KPT, bool F32, bool NN = false>
__global__ void __launch_bounds__(NT) topk_reg_kernel(const void* __restrict__ scores, int Nq,
                                                      int64_t q_pos0, int64_t E, int m, int k,
                                                      int32_t* __restrict__ topk_idx,
                                                      int32_t* __restrict__ topk_cnt) {
  constexpr int NW = NT / 32;
  constexpr int CS = F32 ? 16 : 0;  // shift from a key to its coarse (16-bit) part
  static_assert(KPT <= 32, "a thread's selection is a 32-bit mask");
  __shared__ uint32_t whist[NW * 256];
  __shared__ uint32_t hist1[256], hist2[256], gsum[256];
  __shared__ __align__(16) uint32_t wmax[NW];
  __shared__ uint32_t wa[33], wb[33];
  __shared__ uint32_t cta_val[3];  // this CTA's maximum, keys above T, keys equal to T
  __shared__ uint32_t bcast[2];
  __shared__ int sh_bin;
  __shared__ uint32_t sh_above;
  pdl_trigger();
  pdl_wait();
  const uint32_t C = cluster_nctarank();
  const uint32_t rank = cluster_ctarank();
  const int64_t row = blockIdx.x / C;
  const int64_t t = q_pos0 + (row % Nq);
  const int n = (int)max((int64_t)0, min(E, (t + 1) / m));
  const uint16_t* src = static_cast<const uint16_t*>(scores) + row * E;
  const uint32_t* src32 = static_cast<const uint32_t*>(scores) + row * E;
  int32_t* out = topk_idx + row * (int64_t)k;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (n <= k) {  // uniform over the cluster
    for (int r = (int)rank * NT + tid; r < k; r += (int)C * NT) out[r] = (r < n) ? r : -1;
    if (rank == 0 && tid == 0) topk_cnt[row] = n;
    return;
  }
  // One CTA per row and more rows than SMs (prefill): start the row one wave ahead on its way
  // into L2, so that its CTA does not wait on HBM for its keys.
  if (C == 1 && tid == 0) {
    const int64_t r2 = row + kNumSMs;
    constexpr int kb = F32 ? 4 : 2;
    if (r2 < (int64_t)gridDim.x && (E * kb) % 16 == 0) {
      const int64_t n2 = max((int64_t)0, min(E, (q_pos0 + (r2 % Nq) + 1) / m));
      const char* a2 = static_cast<const char*>(scores) + r2 * E * kb;
      const uint32_t bytes = (uint32_t)((n2 * kb + 15) & ~(int64_t)15);
      if (bytes > 0 && (reinterpret_cast<uintptr_t>(a2) & 15u) == 0) prefetch_l2(a2, bytes);
    }
  }
  // ---- keys of this thread ---------------------------------------------------------------------
  const int seg0 = ((int)rank * NT + tid) * KPT;
  uint32_t key[KPT];
  const uintptr_t sa = F32 ? reinterpret_cast<uintptr_t>(src32) : reinterpret_cast<uintptr_t>(src);
  const bool vec = (sa & 15u) == 0 && seg0 + KPT <= n;
  if constexpr (F32) {
    if (vec) {
#pragma unroll
      for (int q = 0; q < KPT / 4; ++q) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src32 + seg0) + q);
        key[4 * q] = order_key32(v.x);
        key[4 * q + 1] = order_key32(v.y);
        key[4 * q + 2] = order_key32(v.z);
        key[4 * q + 3] = order_key32(v.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < KPT; ++j) key[j] = seg0 + j < n ? order_key32(src32[seg0 + j]) : 0u;
    }
  } else if (vec) {
    uint4 v[KPT / 8];
#pragma unroll
    for (int q = 0; q < KPT / 8; ++q) v[q] = __ldg(reinterpret_cast<const uint4*>(src + seg0) + q);
#pragma unroll
    for (int q = 0; q < KPT / 8; ++q) {
      const uint32_t u[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        key[q * 8 + 2 * h] = NN ? (u[h] & 0xFFFFu) : order_key(u[h] & 0xFFFFu);
        key[q * 8 + 2 * h + 1] = NN ? (u[h] >> 16) : order_key(u[h] >> 16);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      key[j] = seg0 + j < n ? (NN ? (uint32_t)src[seg0 + j] : order_key(src[seg0 + j])) : 0u;
  }
  // slots past the row end hold 0 and are excluded by index, never by value
  // ---- row maximum ----
  uint32_t mx = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) mx = max(mx, key[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) wmax[w] = mx;
  for (int q = tid; q < NW * 256; q += NT) whist[q] = 0u;
  __syncthreads();
  uint32_t row_max = 0;
#pragma unroll
  for (int q = 0; q < NW; q += 4) {  // 16-byte reads of the warps' maxima
    const uint4 v4 = *reinterpret_cast<const uint4*>(&wmax[q]);
    row_max = max(row_max, max(max(v4.x, v4.y), max(v4.z, v4.w)));
  }
  if (C > 1) {
    if (tid == 0) cta_val[0] = row_max;
    cluster_sync();
    if (w == 0) {
      uint32_t v = (uint32_t)lane < C ? dsmem_ld_u32(&cta_val[0], (uint32_t)lane) : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (lane == 0) bcast[0] = v;
    }
    __syncthreads();
    row_max = bcast[0];
  }
  // ---- near-max histogram (one bin per BF16 step below the maximum) ----
  uint32_t* wh = whist + w * 256;
  // The near-max windows hold few keys spread over 255 bins: with the row in one CTA they go
  // straight into one block histogram (whist's first 256 words), which needs no per-warp sum.
  uint32_t* const nh = C == 1 ? whist : wh;
  const uint32_t max_c = row_max >> CS;  // coarse parts of keys and maximum
  // slots past the row end hold key 0, which lies in the window only when the maximum does
  // (max_c < 255): otherwise no test of the position is needed
  if (max_c >= 255u || seg0 + KPT <= n) {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const uint32_t dd = max_c - (key[j] >> CS);
      if (dd < 255u) atomicAdd(&nh[dd], 1u);
    }
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const uint32_t dd = max_c - (key[j] >> CS);
      if (dd < 255u && seg0 + j < n) atomicAdd(&nh[dd], 1u);
    }
  }
  __syncthreads();
  auto sum_hist = [&](uint32_t* hist) {  // per-warp histograms -> hist -> cluster sum in gsum
    reduce_warp_hists<NW>(whist, hist);
    __syncthreads();
    for (int q = tid; q < NW * 256; q += NT) whist[q] = 0u;
    if (C > 1) {
      cluster_sync();
      for (int q = tid; q < 256; q += NT) gsum[q] = cluster_sum(&hist[q], C);
    } else {
      for (int q = tid; q < 256; q += NT) gsum[q] = hist[q];
    }
    __syncthreads();
  };
  auto sum_near = [&](uint32_t* hist) {  // the near-max histogram -> gsum
    if (C == 1) {
      for (int q = tid; q < 256; q += NT) {
        gsum[q] = whist[q];
        whist[q] = 0u;
      }
      __syncthreads();
    } else {
      sum_hist(hist);
    }
  };
  if (C == 1) {
    select_prefix(whist, (uint32_t)k, &sh_bin, &sh_above);  // the block histogram in place
    __syncthreads();
    if (F32 || sh_bin < 0) {  // the searches below count into whist again
      for (int q = tid; q < 256; q += NT) whist[q] = 0u;
      __syncthreads();
    }
  } else {
    sum_hist(hist1);
    select_prefix(gsum, (uint32_t)k, &sh_bin, &sh_above);
    __syncthreads();
  }
  uint32_t Tc, above_c;  // coarse threshold and the count of keys whose coarse part exceeds it
  if (sh_bin >= 0) {
    Tc = max_c - (uint32_t)sh_bin;
    above_c = sh_above;
  } else {
    bool found = false;
    // the histogram arrays of the radix fallback's two digits, alternating with the last one
    // used: every CTA of a cluster has read that one before it arrives at the next barrier
    uint32_t* const hd1 = F32 ? hist2 : hist1;
    uint32_t* const hd2 = F32 ? hist1 : hist2;
    if constexpr (!F32) {
      // second window: the keys 255 .. 509 BF16 steps below the maximum (where the k-th key of a
      // long row usually lies when it is not in the first window)
      const uint32_t in0 = sh_above;  // keys in the first window (fewer than k)
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const uint32_t dd = max_c - key[j];
        if (dd - 255u < 255u && seg0 + j < n) atomicAdd(&nh[dd - 255u], 1u);
      }
      __syncthreads();
      sum_near(hist2);
      select_prefix(gsum, (uint32_t)k - in0, &sh_bin, &sh_above);
      __syncthreads();
      if (sh_bin >= 0) {
        Tc = max_c - 255u - (uint32_t)sh_bin;
        above_c = in0 + sh_above;
        found = true;
      }
    }
    if (!found) {
      // fallback: exact two-digit radix select of the coarse parts on the registers
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        if (seg0 + j < n) atomicAdd(&wh[(key[j] >> CS) >> 8], 1u);
      __syncthreads();
      sum_hist(hd1);
      select_bin(gsum, (uint32_t)k, &sh_bin, &sh_above);
      __syncthreads();
      const uint32_t hi_byte = (uint32_t)sh_bin, above_hi = sh_above;
#pragma unroll
      for (int j = 0; j < KPT; ++j)
        if (seg0 + j < n && (key[j] >> CS >> 8) == hi_byte)
          atomicAdd(&wh[(key[j] >> CS) & 0xFFu], 1u);
      __syncthreads();
      sum_hist(hd2);
      select_bin(gsum, (uint32_t)k - above_hi, &sh_bin, &sh_above);
      __syncthreads();
      Tc = (hi_byte << 8) | (uint32_t)sh_bin;
      above_c = above_hi + sh_above;
    }
  }
  uint32_t T, need_eq;
  if constexpr (F32) {
    // the keys in the coarse bucket Tc: byte 1 of the key, then byte 0 (hist2, then hist1; the
    // last histogram written above was hist1)
    const uint32_t need1 = (uint32_t)k - above_c;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (seg0 + j < n && (key[j] >> 16) == Tc) atomicAdd(&wh[(key[j] >> 8) & 0xFFu], 1u);
    __syncthreads();
    sum_hist(hist2);
    select_bin(gsum, need1, &sh_bin, &sh_above);
    __syncthreads();
    const uint32_t pre = (Tc << 8) | (uint32_t)sh_bin, above2 = sh_above;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (seg0 + j < n && (key[j] >> 8) == pre) atomicAdd(&wh[key[j] & 0xFFu], 1u);
    __syncthreads();
    sum_hist(hist1);
    select_bin(gsum, need1 - above2, &sh_bin, &sh_above);
    __syncthreads();
    T = (pre << 8) | (uint32_t)sh_bin;
    need_eq = need1 - above2 - sh_above;
  } else {
    T = Tc;
    need_eq = (uint32_t)k - above_c;
  }
  // ---- ordered write: bit masks of the selected keys, one scan of their counts; only the set
  // bits are visited ----
  uint32_t gt = 0u, eq = 0u;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    gt |= key[j] > T ? (1u << j) : 0u;
    eq |= key[j] == T ? (1u << j) : 0u;
  }
  {  // keys past the row end are dropped by position
    const int nv = n - seg0;
    const uint32_t valid = nv >= 32 ? 0xFFFFFFFFu : nv <= 0 ? 0u : (1u << nv) - 1u;
    gt &= valid;
    eq &= valid;
  }
  uint32_t gb, eb, tg, te;
  block_scan2((uint32_t)__popc(gt), (uint32_t)__popc(eq), &gb, &eb, &tg, &te, wa, wb);
  if (C > 1) {  // keys of the lower-ranked CTAs of this row
    if (tid == 0) {
      cta_val[1] = tg;
      cta_val[2] = te;
    }
    cluster_sync();
    if (w == 0) {
      uint32_t a = (uint32_t)lane < rank ? dsmem_ld_u32(&cta_val[1], (uint32_t)lane) : 0u;
      uint32_t b = (uint32_t)lane < rank ? dsmem_ld_u32(&cta_val[2], (uint32_t)lane) : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
      }
      if (lane == 0) {
        bcast[0] = a;
        bcast[1] = b;
      }
    }
    cluster_arrive();  // this CTA's remote reads are done; it waits for the others' before exit
    __syncthreads();
    gb += bcast[0];
    eb += bcast[1];
  }
  // this thread takes its lowest-index T-equal keys while the running count is below need_eq
  uint32_t sel = gt;
  for (uint32_t e = eq, take = eb < need_eq ? min(need_eq - eb, (uint32_t)__popc(eq)) : 0u;
       take > 0; --take) {
    const uint32_t low = e & (0u - e);
    sel |= low;
    e ^= low;
  }
  uint32_t pos = gb + min(eb, need_eq);
  while (sel) {
    const int j = __ffs(sel) - 1;
    if (pos < (uint32_t)k) out[pos] = seg0 + j;
    ++pos;
    sel &= sel - 1u;
  }
  if (rank == 0 && tid == 0) topk_cnt[row] = k;
  if (C > 1) cluster_wait();  // no CTA leaves while another may still read its shared memory
}

// Register-resident shapes: keys per CTA = threads x keys per thread.
struct RegShape {
  int nt, kpt;
  int chunk() const { return nt * kpt; }
};
constexpr RegShape kRegShapes[] = {{128, 8}, {256, 16}, {512, 16}, {1024, 16}, {1024, 32}};
constexpr int kMaxRegCluster = 16;

template <int NT, int KPT, bool F32>
cudaError_t launch_reg(const void* scores, int Nq, int64_t q_pos0, int64_t E, int m, int k,
                       int32_t* topk_idx, int32_t* topk_cnt, int64_t rows, int C,
                       cudaStream_t stream, bool nonneg = false) {
  auto kern = nonneg && !F32 ? topk_reg_kernel<NT, KPT, F32, true> : topk_reg_kernel<NT, KPT, F32>;
  if (C > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  ProfScope prof(stream, F32 ? "topk_f32" : "topk");
  return launch_ex(kern, dim3((unsigned)(rows * C)), dim3(NT), 0, stream, (unsigned)C, scores,
                   Nq, q_pos0, E, m, k, topk_idx, topk_cnt);
}

// Whether clusters of C CTAs of this shape can be resident (sizes above 8 are non-portable).
template <int NT, int KPT, bool F32>
bool reg_cluster_fits(int C) {
  if (C <= 8) return true;
  auto kern = topk_reg_kernel<NT, KPT, F32>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)C);
  cfg.blockDim = dim3(NT);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  return nclusters > 0;
}

template <bool F32>
bool reg_fits_query(int shape, int C) {
  switch (shape) {
    case 0: return reg_cluster_fits<128, 8, F32>(C);
    case 1: return reg_cluster_fits<256, 16, F32>(C);
    case 2: return reg_cluster_fits<512, 16, F32>(C);
    case 3: return reg_cluster_fits<1024, 16, F32>(C);
    default: return reg_cluster_fits<1024, 32, F32>(C);
  }
}

// Answers are cached per (key width, shape, cluster size): 0 unknown, 1 fits, 2 does not.
bool reg_fits(int shape, int C, bool f32) {
  static volatile int8_t cache[2][5][kMaxRegCluster + 1] = {};
  if (C <= 8) return true;
  volatile int8_t& c = cache[f32 ? 1 : 0][shape][C];
  if (c == 0) c = (f32 ? reg_fits_query<true>(shape, C) : reg_fits_query<false>(shape, C)) ? 1 : 2;
  return c == 1;
}

// Picks the register-resident shape and cluster size for rows of up to n_max keys: one CTA of
// 32768 keys per row when there are enough rows to fill the GPU; otherwise the smallest chunk
// whose cluster (at most 16 CTAs) covers the row while the grid stays within two CTAs per SM.
// Returns false when no shape covers the row (more than 16 x 32768 keys).
bool pick_reg(int64_t rows, int64_t n_max, int* shape, int* C, bool f32) {
  constexpr int nshapes = (int)(sizeof(kRegShapes) / sizeof(kRegShapes[0]));
  if (n_max <= kRegShapes[nshapes - 1].chunk() && rows >= kNumSMs) {
    // enough rows to fill the GPU: one CTA per row, the smallest one that holds the row
    int i = 0;
    while (kRegShapes[i].chunk() < n_max) ++i;
    *shape = i;
    *C = 1;
    return true;
  }
  int best = -1, best_c = 0;
  for (int i = 0; i < nshapes; ++i) {
    const int64_t c = (n_max + kRegShapes[i].chunk() - 1) / kRegShapes[i].chunk();
    if (c > kMaxRegCluster || !reg_fits(i, (int)max((int64_t)1, c), f32)) continue;
    best = i;
    best_c = (int)max((int64_t)1, c);
    if (rows * best_c <= 2 * kNumSMs) break;
  }
  if (best < 0) return false;
  *shape = best;
  *C = best_c;
  return true;
}

template <int NT>
cudaError_t launch_topk_t(const uint16_t* scores, int Nq, int64_t q_pos0, int64_t E, int m, int k,
                          int32_t* topk_idx, int32_t* topk_cnt, int64_t rows, int64_t n_max,
                          int C, int chunk_cap, cudaStream_t stream) {
  auto kern = topk_kernel<NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       chunk_cap * 2);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  int cap = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // Clusters of 16 are a non-portable size: fall back to 8 if this GPU cannot hold one.
  for (;; C >>= 1) {
    const int64_t chunk = (n_max + C - 1) / C;
    cap = (n_max > k && chunk <= chunk_cap) ? (int)chunk : 0;
    cfg.dynamicSmemBytes = (size_t)cap * 2;
    cfg.gridDim = dim3((unsigned)C, (unsigned)rows, 1);
    attr[0].val.clusterDim.x = (unsigned)C;
    int nclusters = 0;
    if (C <= 8 || (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) == cudaSuccess &&
                   nclusters > 0))
      break;
    (void)cudaGetLastError();
  }
  ProfScope prof(stream, "topk");
  return cudaLaunchKernelEx(&cfg, kern, scores, Nq, q_pos0, E, m, k, cap, topk_idx, topk_cnt);
}

template <bool F32>
cudaError_t launch_reg_shape(int shape, const void* scores, int Nq, int64_t q_pos0, int64_t E,
                             int m, int k, int32_t* topk_idx, int32_t* topk_cnt, int64_t rows,
                             int C, cudaStream_t stream, bool nonneg = false) {
  switch (shape) {
    case 0:
      return launch_reg<128, 8, F32>(scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows, C,
                                     stream, nonneg);
    case 1:
      return launch_reg<256, 16, F32>(scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows, C,
                                      stream, nonneg);
    case 2:
      return launch_reg<512, 16, F32>(scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows, C,
                                      stream, nonneg);
    case 3:
      return launch_reg<1024, 16, F32>(scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows, C,
                                       stream, nonneg);
    default:
      return launch_reg<1024, 32, F32>(scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows, C,
                                       stream, nonneg);
  }
}

}  // namespace

cudaError_t launch_topk(const uint16_t* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                        int k, int32_t* topk_idx, int32_t* topk_cnt, cudaStream_t stream,
                        bool nonneg) {
  const int64_t rows = (int64_t)B * Nq;
  if (rows <= 0) return cudaSuccess;
  int64_t n_max = min(E, (q_pos0 + Nq) / m);
  if (n_max < 0) n_max = 0;
  int shape = 0, C = 1;
  if (pick_reg(rows, n_max, &shape, &C, false))
    return launch_reg_shape<false>(shape, scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows,
                                   C, stream, nonneg);
  // rows longer than 16 x 32768 keys: clusters of up to 16 CTAs staging their chunks in
  // shared memory
  int Cs = 1;
  while (Cs < 16 && (n_max + Cs - 1) / Cs > kMaxChunkKeys) Cs <<= 1;
  return launch_topk_t<kClusterThreads>(scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows,
                                        n_max, Cs, kMaxChunkKeys, stream);
}

cudaError_t launch_topk_f32(const float* scores, int B, int Nq, int64_t q_pos0, int64_t E, int m,
                            int k, int32_t* topk_idx, int32_t* topk_cnt, cudaStream_t stream) {
  const int64_t rows = (int64_t)B * Nq;
  if (rows <= 0) return cudaSuccess;
  int64_t n_max = min(E, (q_pos0 + Nq) / m);
  if (n_max < 0) n_max = 0;
  int shape = 0, C = 1;
  if (!pick_reg(rows, n_max, &shape, &C, true)) return cudaErrorInvalidValue;
  return launch_reg_shape<true>(shape, scores, Nq, q_pos0, E, m, k, topk_idx, topk_cnt, rows, C,
                                stream);
}

}  // namespace csa
