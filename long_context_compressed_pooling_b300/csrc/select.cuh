// Selection helpers shared by the top-k kernels (topk.cu) and the fused decode kernel
// (decode.cu): order-preserving keys for BF16 / FP32 scores, 256-bin histogram searches, a
// block-wide scan of two counters, and cluster-wide reductions through distributed shared
// memory.
#pragma once

#include "common.cuh"

namespace csa {

CSA_DEV uint32_t order_key(uint32_t bits) {
  if (bits == 0x8000u) bits = 0u;  // -0 counts as +0
  return (bits & 0x8000u) ? (~bits & 0xFFFFu) : (bits | 0x8000u);
}

// FP32 scores: the same order-preserving map on 32-bit patterns.
CSA_DEV uint32_t order_key32(uint32_t bits) {
  if (bits == 0x80000000u) bits = 0u;  // -0 counts as +0
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// Sums the per-warp histograms whist[NW][256] into hist[256] (all threads call it).
template <int NW>
CSA_DEV void reduce_warp_hists(const uint32_t* whist, uint32_t* hist) {
  for (int q = threadIdx.x; q < 256; q += blockDim.x) {
    uint32_t s = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += whist[w * 256 + q];
    hist[q] = s;
  }
}

// Finds the bin b with count(bins > b) < need <= count(bins >= b) over 256 bins; writes the bin
// and count(bins > b). Executed by warp 0.
CSA_DEV void select_bin(const uint32_t* hist, uint32_t need, int* out_bin, uint32_t* out_above) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t local[8];
    uint32_t tot = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      local[q] = hist[255 - (lane * 8 + q)];
      tot += local[q];
    }
    uint32_t inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
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

// Finds the first bin b (ascending) with prefix(b-1) < need <= prefix(b) over bins [0, 255);
// writes b and prefix(b-1), or bin -1 and the total of the 255 bins when they hold fewer than
// `need`. Warp 0 only.
CSA_DEV void select_prefix(const uint32_t* hist, uint32_t need, int* out_bin, uint32_t* out_before) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    uint32_t local[8];
    uint32_t tot = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int bin = lane * 8 + q;
      local[q] = bin < 255 ? hist[bin] : 0u;
      tot += local[q];
    }
    uint32_t inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const uint32_t exc = inc - tot;
    if (lane == 31 && inc < need) {
      *out_bin = -1;
      *out_before = inc;
    }
    if (exc < need && need <= inc) {
      uint32_t run = exc;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (run < need && need <= run + local[q]) {
          *out_bin = lane * 8 + q;
          *out_before = run;
        }
        run += local[q];
      }
    }
  }
}

// Largest 32-bit word at `p` over CTAs 0..n-1 of the cluster (n <= 16).
CSA_DEV uint32_t cluster_max(const uint32_t* p, uint32_t n) {
  uint32_t v[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) v[c] = (uint32_t)c < n ? dsmem_ld_u32(p, (uint32_t)c) : 0u;
  uint32_t m = 0;
#pragma unroll
  for (int c = 0; c < 16; ++c) m = max(m, v[c]);
  return m;
}

// Block-wide exclusive scan of two counters (one pair per thread); also returns the totals.
CSA_DEV void block_scan2(uint32_t a, uint32_t b, uint32_t* ex_a, uint32_t* ex_b, uint32_t* tot_a,
                         uint32_t* tot_b, uint32_t* wa, uint32_t* wb) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t va = __shfl_up_sync(0xffffffffu, ia, o);
    const uint32_t vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += va;
      ib += vb;
    }
  }
  if (lane == 31) {
    wa[w] = ia;
    wb[w] = ib;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    const uint32_t xa = lane < nw ? wa[lane] : 0u, xb = lane < nw ? wb[lane] : 0u;
    uint32_t sa = xa, sb = xb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t va = __shfl_up_sync(0xffffffffu, sa, o);
      const uint32_t vb = __shfl_up_sync(0xffffffffu, sb, o);
      if (lane >= o) {
        sa += va;
        sb += vb;
      }
    }
    if (lane < nw) {
      wa[lane] = sa - xa;
      wb[lane] = sb - xb;
    }
    if (lane == nw - 1) {
      wa[32] = sa;
      wb[32] = sb;
    }
  }
  __syncthreads();
  *ex_a = wa[w] + ia - a;
  *ex_b = wb[w] + ib - b;
  *tot_a = wa[32];
  *tot_b = wb[32];
  __syncthreads();  // wa / wb are reused by the next call
}

// Sum of the 32-bit word at `p` over CTAs 0..n-1 of the cluster (n <= 16): all remote loads are
// issued before any of them is consumed.
CSA_DEV uint32_t cluster_sum(const uint32_t* p, uint32_t n) {
  uint32_t v[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) v[c] = (uint32_t)c < n ? dsmem_ld_u32(p, (uint32_t)c) : 0u;
  uint32_t s = 0;
#pragma unroll
  for (int c = 0; c < 16; ++c) s += v[c];
  return s;
}

}  // namespace csa
