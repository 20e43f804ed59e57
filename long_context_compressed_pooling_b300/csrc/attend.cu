// CSA sparse attention and HCA dense attention over compressed entries plus a sliding window:
// the split-K mma.sync flash-decode kernel (head dim 64, one query per sequence), the split
// planner, the workspace merge and the dispatcher (head dim 128 goes to the tcgen05 kernel in
// attend_tc.cu, head dim 64 prefill to the packed tcgen05 kernel in attend_pk.cu).
//
// Lighthouse "deep deepseek v4 release" 八.3: CSA attends to the top-k selected compressed
// entries plus a sliding-window branch of n_win raw tokens; HCA attends densely to every
// compressed entry (m' = 128) plus the same window. One softmax spans the entries and the window
// tokens of a query; logits are q.k (the 1/sqrt(d) is folded into q).
//
// MQA layout: all H query heads of a token share one K/V head, so the heads form the M side of
// the contraction. A CTA owns one query token and up to 64 heads (16 per warp) and walks a
// range of 64-key chunks of that token's key list: the chunk's K and V rows are gathered with
// 16-byte cp.async into XOR-swizzled shared memory through a 3-stage pipeline, QK^T and PV run
// on the tensor cores, and the softmax is an online (running max / sum) softmax in registers.
// When a token's keys are split over several CTAs (decode), the splits of one token form a
// thread-block cluster: each CTA parks its (max, sum, unnormalised O) in its own shared memory
// and, after a hardware cluster barrier, merges a slice of the heads by reading every split's
// partials through distributed shared memory. Very small batches that need more than 16 splits
// per token merge through the workspace with a separate kernel instead.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kKC = 64;      // keys per chunk
constexpr int kStages = 3;   // cp.async pipeline depth
constexpr int kMaxClusterSplits = 16;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const uint16_t* q;
  const uint16_t* k_cmp;
  const uint16_t* v_cmp;
  const int32_t* topk_idx;
  const int32_t* topk_cnt;
  const uint16_t* k_raw;
  const uint16_t* v_raw;
  uint16_t* out;
  float* lse;
  float* ws_o;   // [n_splits, tokens, H, D] unnormalised partial outputs (workspace merge)
  float* ws_ml;  // [n_splits, tokens, H, 2] running max and sum
  int64_t E, N, q_pos0;
  int k, m, W, Nq, H, n_splits, tokens;
  int sparse;
  int cluster_merge;  // splits of a token form a cluster and merge through DSMEM
  uint32_t* status;
};

CSA_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
CSA_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
CSA_DEV void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32"
      " {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int D>
constexpr size_t attend_smem_bytes() {
  return (size_t)kStages * 2 * kKC * D * 2 + kStages * kKC;
}

template <int D, int NW>
__global__ void __launch_bounds__(NW * 32) attend_kernel(const AttnParams p) {
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  constexpr int NT = 32 * NW;
  constexpr int ROWS = 16 * NW;     // heads of this CTA
  constexpr int PSTRIDE = D + 4;    // padded row stride of the parked partial outputs
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);                   // [kStages][kKC][D]
  uint16_t* Vs = Ks + kStages * kKC * D;                              // [kStages][kKC][D]
  uint8_t* kmask = reinterpret_cast<uint8_t*>(Vs + kStages * kKC * D);  // [kStages][kKC]

  pdl_trigger();
  pdl_wait();
  const int split = p.cluster_merge ? (int)cluster_ctarank() : blockIdx.x;
  const int64_t tok = blockIdx.y;
  const int h_base = blockIdx.z * ROWS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;

  const int64_t b = tok / p.Nq;
  const int64_t t = p.q_pos0 + tok % p.Nq;
  int64_t n_sel;
  if (p.sparse) {
    n_sel = p.topk_cnt[tok];
    if (n_sel < 0 || n_sel > p.k) {
      if (threadIdx.x == 0) atomicOr(p.status, kFlagBadIndex);
      n_sel = n_sel < 0 ? 0 : p.k;
    }
  } else {
    n_sel = max((int64_t)0, min(p.E, (t + 1) / p.m));
  }
  const int64_t w0 = max((int64_t)0, t - p.W + 1);
  const int64_t n_keys = n_sel + (p.W > 0 ? (t - w0 + 1) : 0);
  const int64_t n_chunks = (n_keys + kKC - 1) / kKC;
  const int64_t c_begin = n_chunks * split / p.n_splits;
  const int64_t c_end = n_chunks * (split + 1) / p.n_splits;

  auto load_chunk = [&](int64_t c, int st) {
    uint16_t* kd = Ks + st * kKC * D;
    uint16_t* vd = Vs + st * kKC * D;
    for (int x = threadIdx.x; x < kKC * CPR; x += NT) {
      const int r = x / CPR, cc = x % CPR;
      const int64_t key = c * kKC + r;
      const uint16_t* ks = p.k_raw;
      const uint16_t* vs = p.v_raw;
      bool valid = key < n_keys;
      if (valid) {
        if (key < n_sel) {
          const int64_t j = p.sparse ? (int64_t)p.topk_idx[tok * p.k + key] : key;
          if (j < 0 || j >= p.E) {
            valid = false;
            if (cc == 0) atomicOr(p.status, kFlagBadIndex);
          } else {
            ks = p.k_cmp + (b * p.E + j) * D;
            vs = p.v_cmp + (b * p.E + j) * D;
          }
        } else {
          const int64_t u = w0 + (key - n_sel);
          ks = p.k_raw + (b * p.N + u) * D;
          vs = p.v_raw + (b * p.N + u) * D;
        }
      }
      const int phys = r * CPR + (cc ^ (r & 7));
      cp_async_16(kd + phys * 8, valid ? ks + cc * 8 : p.k_raw, valid ? 16u : 0u);
      cp_async_16(vd + phys * 8, valid ? vs + cc * 8 : p.v_raw, valid ? 16u : 0u);
      if (cc == 0) kmask[st * kKC + r] = valid ? 1 : 0;
    }
  };

  // Put the first chunks in flight before anything else.
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (c_begin + s < c_end) load_chunk(c_begin + s, s);
    cp_async_commit();
  }

  // Q fragments (rows h0 = h_base + warp*16 + g and h0 + 8), A layout of m16n8k16.
  const int h0 = h_base + warp * 16 + g, h1 = h0 + 8;
  uint32_t qa[D / 16][4];
  {
    const uint16_t* q0 = p.q + (tok * p.H + h0) * D;
    const uint16_t* q1 = p.q + (tok * p.H + h1) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c0 = kk * 16 + 2 * tq;
      qa[kk][0] = h0 < p.H ? *reinterpret_cast<const uint32_t*>(q0 + c0) : 0u;
      qa[kk][1] = h1 < p.H ? *reinterpret_cast<const uint32_t*>(q1 + c0) : 0u;
      qa[kk][2] = h0 < p.H ? *reinterpret_cast<const uint32_t*>(q0 + c0 + 8) : 0u;
      qa[kk][3] = h1 < p.H ? *reinterpret_cast<const uint32_t*>(q1 + c0 + 8) : 0u;
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int mi = lane >> 3, rr = lane & 7;

  for (int64_t c = c_begin; c < c_end; ++c) {
    const int it = (int)(c - c_begin);
    if (c + kStages - 1 < c_end) load_chunk(c + kStages - 1, (it + kStages - 1) % kStages);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const int st = it % kStages;
    const uint32_t kbase = smem_addr(Ks + st * kKC * D);
    const uint32_t vbase = smem_addr(Vs + st * kKC * D);
    const uint8_t* msk = kmask + st * kKC;

    // ---- S = Q K^T over 64 keys ----
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int r = 16 * pp + (mi >> 1) * 8 + rr;
        const int cc = 2 * kk + (mi & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + (uint32_t)((r * CPR + (cc ^ (r & 7))) * 16), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * pp], qa[kk], b0, b1);
        mma_bf16_16816(s[2 * pp + 1], qa[kk], b2, b3);
      }
    }
    // ---- mask + online softmax ----
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int col = nt * 8 + 2 * tq;
      if (!msk[col]) s[nt][0] = s[nt][2] = -INFINITY;
      if (!msk[col + 1]) s[nt][1] = s[nt][3] = -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
#pragma unroll
    for (int o2 = 1; o2 < 4; o2 <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0;
    const float base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float corr0 = exp2f((m0 - base0) * kLog2e), corr1 = exp2f((m1 - base1) * kLog2e);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = exp2f((s[nt][0] - base0) * kLog2e);
      const float p1 = exp2f((s[nt][1] - base0) * kLog2e);
      const float p2 = exp2f((s[nt][2] - base1) * kLog2e);
      const float p3 = exp2f((s[nt][3] - base1) * kLog2e);
      rs0 += p0 + p1;
      rs1 += p2 + p3;
      const int kk2 = nt >> 1, hi = nt & 1;
      pa[kk2][hi * 2 + 0] = pack_bf16x2(p0, p1);
      pa[kk2][hi * 2 + 1] = pack_bf16x2(p2, p3);
    }
    l0 = l0 * corr0 + rs0;
    l1 = l1 * corr1 + rs1;
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= corr0;
      o[i][1] *= corr0;
      o[i][2] *= corr1;
      o[i][3] *= corr1;
    }
    // ---- O += P V ----
#pragma unroll
    for (int kk2 = 0; kk2 < 4; ++kk2) {
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int r = 16 * kk2 + (mi & 1) * 8 + rr;
        const int cc = 2 * dp + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + (uint32_t)((r * CPR + (cc ^ (r & 7))) * 16), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa[kk2], b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa[kk2], b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- finish: quad-reduce the row sums, then store / park / merge ----
#pragma unroll
  for (int o2 = 1; o2 < 4; o2 <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
  }
  if (p.n_splits == 1) {
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      const int d0 = dt * 8 + 2 * tq;
      if (h0 < p.H)
        *reinterpret_cast<uint32_t*>(p.out + (tok * p.H + h0) * D + d0) =
            pack_bf16x2(o[dt][0] * inv0, o[dt][1] * inv0);
      if (h1 < p.H)
        *reinterpret_cast<uint32_t*>(p.out + (tok * p.H + h1) * D + d0) =
            pack_bf16x2(o[dt][2] * inv1, o[dt][3] * inv1);
    }
    if (p.lse != nullptr && tq == 0) {
      if (h0 < p.H) p.lse[tok * p.H + h0] = l0 > 0.f ? m0 + logf(l0) : -INFINITY;
      if (h1 < p.H) p.lse[tok * p.H + h1] = l1 > 0.f ? m1 + logf(l1) : -INFINITY;
    }
    return;
  }
  if (!p.cluster_merge) {
    const int64_t sb = ((int64_t)split * p.tokens + tok) * p.H;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      const int d0 = dt * 8 + 2 * tq;
      if (h0 < p.H)
        *reinterpret_cast<float2*>(p.ws_o + (sb + h0) * D + d0) = make_float2(o[dt][0], o[dt][1]);
      if (h1 < p.H)
        *reinterpret_cast<float2*>(p.ws_o + (sb + h1) * D + d0) = make_float2(o[dt][2], o[dt][3]);
    }
    if (tq == 0) {
      if (h0 < p.H) *reinterpret_cast<float2*>(p.ws_ml + (sb + h0) * 2) = make_float2(m0, l0);
      if (h1 < p.H) *reinterpret_cast<float2*>(p.ws_ml + (sb + h1) * 2) = make_float2(m1, l1);
    }
    return;
  }
  // Cluster merge: park this split's partials in shared memory (the pipeline buffers are free).
  float* po = reinterpret_cast<float*>(smem);  // [ROWS][PSTRIDE]
  float* pml = po + ROWS * PSTRIDE;            // [ROWS][2]
  const int r0 = warp * 16 + g, r1 = r0 + 8;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int d0 = dt * 8 + 2 * tq;
    *reinterpret_cast<float2*>(po + r0 * PSTRIDE + d0) = make_float2(o[dt][0], o[dt][1]);
    *reinterpret_cast<float2*>(po + r1 * PSTRIDE + d0) = make_float2(o[dt][2], o[dt][3]);
  }
  if (tq == 0) {
    *reinterpret_cast<float2*>(pml + r0 * 2) = make_float2(m0, l0);
    *reinterpret_cast<float2*>(pml + r1 * 2) = make_float2(m1, l1);
  }
  __syncthreads();
  cluster_sync();
  // This CTA merges rows [rb, re) of the head group, D/4 float4 columns per row.
  const int S = p.n_splits;
  const int rows_per = (ROWS + S - 1) / S;
  const int rb = split * rows_per, re = min(ROWS, rb + rows_per);
  constexpr int C4 = D / 4;
  for (int x = threadIdx.x; x < (re - rb) * C4; x += NT) {
    const int row = rb + x / C4, c4 = x % C4;
    const int h = h_base + row;
    if (h >= p.H) continue;
    float2 ml[kMaxClusterSplits];
#pragma unroll
    for (int sp = 0; sp < kMaxClusterSplits; ++sp)
      ml[sp] = sp < S ? dsmem_ld_f32x2(pml + row * 2, sp) : make_float2(-INFINITY, 0.f);
    float M = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kMaxClusterSplits; ++sp) M = fmaxf(M, ml[sp].x);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
      float4 v[kMaxClusterSplits];
#pragma unroll
      for (int sp = 0; sp < kMaxClusterSplits; ++sp)
        v[sp] = sp < S ? dsmem_ld_f32x4(po + row * PSTRIDE + c4 * 4, sp)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
        if (ml[sp].x == -INFINITY) continue;
        const float w = expf(ml[sp].x - M);
        L += w * ml[sp].y;
        acc.x += w * v[sp].x;
        acc.y += w * v[sp].y;
        acc.z += w * v[sp].z;
        acc.w += w * v[sp].w;
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.out + (tok * p.H + h) * D + c4 * 4) = pk;
    if (p.lse != nullptr && c4 == 0) p.lse[tok * p.H + h] = L > 0.f ? M + logf(L) : -INFINITY;
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

// Combines workspace split-K partials: out = sum_s w_s O_s / sum_s w_s l_s, w_s = exp(m_s - max m).
// One CTA of 8 warps per (token, head). Warp g takes splits g, g + 8, ... in batches of eight,
// all of whose (max, sum) pairs and partial rows are loaded before any is used, and keeps its own
// running maximum (an online merge); the eight warp results are combined through shared memory.
// Every load of a batch is in flight at once, so a merge of up to 64 splits costs one round trip.
constexpr int kMergeWarps = 8, kMergeBatch = 8;
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const float* __restrict__ ws_o,
                                                                 const float* __restrict__ ws_ml,
                                                                 int n_splits, int64_t tokens,
                                                                 int H, uint16_t* out, float* lse) {
  constexpr int PER = D / 32;  // 4 (D = 128) or 2 (D = 64) consecutive floats per lane
  __shared__ float s_acc[kMergeWarps][D];
  __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
  pdl_trigger();
  pdl_wait();
  const int64_t th = blockIdx.x;  // tok * H + h
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t stride = tokens * H;
  float Mw = -INFINITY, Lw = 0.f, acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int s0 = w; s0 < n_splits; s0 += kMergeWarps * kMergeBatch) {
    float2 ml[kMergeBatch];
    float o[kMergeBatch][PER];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int sp = s0 + u * kMergeWarps;
      ml[u] = make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int i = 0; i < PER; ++i) o[u][i] = 0.f;
      if (sp < n_splits) {
        ml[u] = *reinterpret_cast<const float2*>(ws_ml + ((int64_t)sp * stride + th) * 2);
        const float* src = ws_o + ((int64_t)sp * stride + th) * D + lane * PER;
        if constexpr (PER == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          o[u][0] = v.x;
          o[u][1] = v.y;
          o[u][2] = v.z;
          o[u][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          o[u][0] = v.x;
          o[u][1] = v.y;
        }
      }
    }
    float bm = Mw;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) bm = fmaxf(bm, ml[u].x);
    if (bm == -INFINITY) continue;
    const float sc = Mw == -INFINITY ? 0.f : expf(Mw - bm);
    Lw *= sc;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] *= sc;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float wt = ml[u].x == -INFINITY ? 0.f : expf(ml[u].x - bm);
      Lw = fmaf(wt, ml[u].y, Lw);
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(wt, o[u][i], acc[i]);
    }
    Mw = bm;
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) s_acc[w][lane * PER + i] = acc[i];
  if (lane == 0) {
    s_m[w] = Mw;
    s_l[w] = Lw;
  }
  __syncthreads();
  if (threadIdx.x < D / 2) {
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < kMergeWarps; ++g) M = fmaxf(M, s_m[g]);
    float L = 0.f, a0 = 0.f, a1 = 0.f;
    if (M != -INFINITY) {
      const int d = 2 * threadIdx.x;
#pragma unroll
      for (int g = 0; g < kMergeWarps; ++g) {
        const float wt = s_m[g] == -INFINITY ? 0.f : expf(s_m[g] - M);
        L = fmaf(wt, s_l[g], L);
        a0 = fmaf(wt, s_acc[g][d], a0);
        a1 = fmaf(wt, s_acc[g][d + 1], a1);
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    *reinterpret_cast<uint32_t*>(out + th * D + 2 * threadIdx.x) = pack_bf16x2(a0 * inv, a1 * inv);
    if (lse != nullptr && threadIdx.x == 0) lse[th] = L > 0.f ? M + logf(L) : -INFINITY;
  }
}

struct SplitPlan {
  int n_splits;
  int cluster;  // 1: merge inside a cluster of n_splits CTAs
};

// Splits of a token's key chunks over CTAs. The mma.sync kernel (64-key chunks, two CTAs per SM)
// aims at 2 x 148 CTAs; the tcgen05 kernel (128-key chunks, one CTA per SM) at one wave of 148.
SplitPlan plan_splits(int tokens, int H, int64_t max_keys, int d) {
  const bool tc = d == 128;
  const int64_t kc = tc ? attend_tc_chunk_keys() : kKC;
  const int64_t groups = (H + 63) / 64;
  const int64_t chunks = (max_keys + kc - 1) / kc;
  const int64_t units = (int64_t)tokens * groups;
  const int64_t target = tc ? (int64_t)kNumSMs : (int64_t)kNumSMs * 2;
  if (units >= target || chunks <= 1) return {1, 0};
  int64_t s = tc ? target / units : (target + units - 1) / units;
  if (s > chunks) s = chunks;
  if (s <= 1) return {1, 0};
  if (s <= kMaxClusterSplits) return {(int)s, 1};
  return {(int)s, 0};
}

template <int D, int NW>
cudaError_t launch_attend_t(AttnParams prm, int groups, cudaStream_t stream) {
  const size_t smem = attend_smem_bytes<D>();
  auto kern = attend_kernel<D, NW>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (prm.cluster_merge && prm.n_splits > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)prm.n_splits, (unsigned)prm.tokens, (unsigned)groups);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = prm.cluster_merge ? (unsigned)prm.n_splits : 1u;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (prm.cluster_merge && prm.n_splits > 8) {
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess || nclusters == 0) {
      (void)cudaGetLastError();
      return cudaErrorNotSupported;  // caller falls back to the workspace merge
    }
  }
  {
    ProfScope prof(stream, prm.sparse ? "csa_attend" : "hca_attend");
    e = cudaLaunchKernelEx(&cfg, kern, prm);
  }
  if (e != cudaSuccess || prm.n_splits == 1 || prm.cluster_merge) return e;
  ProfScope prof(stream, "lse_merge");
  return launch_ex(merge_kernel<D>, dim3((unsigned)((int64_t)prm.tokens * prm.H)),
                   dim3(kMergeWarps * 32), 0, stream, 1, (const float*)prm.ws_o, (const float*)prm.ws_ml, prm.n_splits,
                   (int64_t)prm.tokens, prm.H, prm.out, prm.lse);
}

template <int D>
cudaError_t launch_d(AttnParams prm, int groups, int nw, cudaStream_t stream) {
  if (nw == 1) return launch_attend_t<D, 1>(prm, groups, stream);
  if (nw == 2) return launch_attend_t<D, 2>(prm, groups, stream);
  return launch_attend_t<D, 4>(prm, groups, stream);
}

}  // namespace

int plan_attend_splits(int tokens, int H, int d, int64_t max_keys) {
  return plan_splits(tokens, H, max_keys, d).n_splits;
}

size_t attend_workspace_bytes(int tokens, int H, int d, int64_t max_keys) {
  // The workspace covers the non-cluster merge, which is also the fallback of the cluster one.
  const int s = plan_splits(tokens, H, max_keys, d).n_splits;
  if (s <= 1) return 0;
  return (size_t)s * tokens * H * (size_t)(d + 2) * sizeof(float);
}

namespace {
cudaError_t launch_merge(int D, const float* ws_o, const float* ws_ml, int n_splits, int tokens,
                         int H, uint16_t* out, float* lse, cudaStream_t stream) {
  ProfScope prof(stream, "lse_merge");
  const dim3 grid((unsigned)((int64_t)tokens * H));
  if (D == 128)
    return launch_ex(merge_kernel<128>, grid, dim3(kMergeWarps * 32), 0, stream, 1, ws_o, ws_ml,
                     n_splits, (int64_t)tokens, H, out, lse);
  return launch_ex(merge_kernel<64>, grid, dim3(kMergeWarps * 32), 0, stream, 1, ws_o, ws_ml,
                   n_splits, (int64_t)tokens, H, out, lse);
}
}  // namespace

cudaError_t launch_attend(const AttendArgs& a, int64_t max_keys, void* ws, uint32_t* status,
                          cudaStream_t stream) {
  const int tokens = a.B * a.Nq;
  if (tokens == 0) return cudaSuccess;
  if (a.d != 128 && a.d != 64) return cudaErrorInvalidValue;
  if (a.paged && a.d != 128) return cudaErrorInvalidValue;  // paged reads: tcgen05 kernel only
  if (a.d == 64 && a.Nq > 1) return launch_attend_pk(a, status, stream);  // prefill
  const SplitPlan sp = plan_splits(tokens, a.H, max_keys, a.d);
  float* ws_o = reinterpret_cast<float*>(ws);
  float* ws_ml = ws_o + (size_t)sp.n_splits * tokens * a.H * a.d;
  if (a.d == 128) {
    // tcgen05 kernel
    int cluster = sp.cluster;
    cudaError_t e = launch_attend_tc(a, sp.n_splits, cluster, ws_o, ws_ml, status, stream);
    if (e == cudaErrorNotSupported && cluster) {
      cluster = 0;
      e = launch_attend_tc(a, sp.n_splits, 0, ws_o, ws_ml, status, stream);
    }
    if (e != cudaSuccess || sp.n_splits == 1 || cluster) return e;
    return launch_merge(a.d, ws_o, ws_ml, sp.n_splits, tokens, a.H, a.out, a.lse, stream);
  }
  AttnParams prm;
  prm.q = a.q;
  prm.k_cmp = a.k_cmp;
  prm.v_cmp = a.v_cmp;
  prm.topk_idx = a.topk_idx;
  prm.topk_cnt = a.topk_cnt;
  prm.k_raw = a.k_raw;
  prm.v_raw = a.v_raw;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.E = a.E;
  prm.N = a.N;
  prm.q_pos0 = a.q_pos0;
  prm.k = a.k;
  prm.m = a.m;
  prm.W = a.W;
  prm.Nq = a.Nq;
  prm.H = a.H;
  prm.tokens = tokens;
  prm.sparse = a.topk_idx != nullptr;
  prm.status = status;
  prm.n_splits = sp.n_splits;
  prm.cluster_merge = sp.cluster;
  prm.ws_o = ws_o;
  prm.ws_ml = ws_ml;
  const int groups = (a.H + 63) / 64;
  const int nw = a.H >= 64 ? 4 : (a.H + 15) / 16 >= 3 ? 4 : (a.H + 15) / 16;
  cudaError_t e = launch_d<64>(prm, groups, nw, stream);
  if (e == cudaErrorNotSupported && prm.cluster_merge) {
    prm.cluster_merge = 0;
    e = launch_d<64>(prm, groups, nw, stream);
  }
  return e;
}

}  // namespace csa
