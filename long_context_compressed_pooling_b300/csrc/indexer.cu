// Lightning Indexer scores on the 5th-generation tensor cores (tcgen05, FP4).
//
// 9fzt.com DeepSeek-V4 summary, item 4: the CSA indexer's QK path runs in FP4 and its scores
// are reduced from FP32 to BF16 before the top-k selector. Lighthouse "deep deepseek v4
// release" 八.7: the indexer keeps its own compressed keys.
//   s[b,i,j] = bf16_rne( sum_h max(0, q_I[b,i,h] . k_I[b,j]) )
// with q_I, k_I block-scaled FP4 vectors (e2m1 codes, one UE8M0 scale per 32 elements).
//
// Layout of the contraction. A = the entries' FP4 index keys (M = 128 entries per tile,
// K = 64 e2m1 values = 32 bytes per row, TMA-loaded with the 32-byte swizzle). B = the queries,
// one B row per (query, head, 32-element block): the row holds that block's codes and zeros
// elsewhere, so D[j, (q,h,blk)] is the UNSCALED partial dot product of one scale block. The
// MMA runs kind::mxf4 with every scale factor set to 1.0; the real UE8M0 scales are applied in
// the epilogue as exact power-of-two multiplies. Partial sums of e2m1 products are multiples of
// 1/4 below 2^11, so the tensor core's fp32 accumulation is exact, and the epilogue's scaled
// sums stay exact for the scale range the workloads use (2^-4..2^0): the BF16 rounding is then
// the only rounding, as the method specifies.
//
// Warp roles (192 threads): warp 0 issues TMA loads into a 4-stage ring, warp 1 allocates
// tensor memory and issues one MMA per 128-entry tile into a double-buffered accumulator,
// warps 2-5 drain the accumulator (tcgen05.ld), apply scales / ReLU / head sum / BF16 rounding
// and store the scores. Every mbarrier wait is bounded (kFlagTimeout on expiry).
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kTileM = 128;
constexpr int kStages = 4;
constexpr int kRowBytes = 32;
constexpr int kATileBytes = kTileM * kRowBytes;
constexpr int kThreads = 192;
constexpr int kMaxCols = 64;
constexpr int kSfCols = 16;  // tensor-memory columns filled with scale 1.0 for each of A and B

struct IdxParams {
  const uint8_t* qi_codes;   // [B, Nq, H_I, NB*16]
  const uint8_t* qi_scales;  // [B, Nq, H_I, NB]
  const uint8_t* ki_scales;  // [B, E, NB]
  uint16_t* scores;          // [B, Nq, E]
  int64_t q_pos0, E;
  int Nq, m, QN, ncols, n_splits, tmem_cols;
  uint32_t* status;
};

constexpr size_t kSmemBytes = 1024 /*align slack*/ + kStages * kATileBytes +
                              kMaxCols * kRowBytes + kMaxCols * sizeof(float) + 256;

// H_I heads, NB = d_I / 32 scale blocks per vector; CPQ = H_I * NB MMA columns per query.
template <int H_I, int NB>
__global__ void __launch_bounds__(kThreads) indexer_kernel(const __grid_constant__ CUtensorMap kmap,
                                                           const IdxParams p) {
  constexpr int CPQ = H_I * NB;
  static_assert(16 % CPQ == 0, "columns per query must divide 16");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* atiles = base;                                   // kStages x 4096, 1024-aligned
  uint8_t* btile = atiles + kStages * kATileBytes;          // ncols x 32, 1024-aligned
  float* qscale = reinterpret_cast<float*>(btile + kMaxCols * kRowBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(qscale + kMaxCols);
  uint64_t* full = bars;                 // [kStages]
  uint64_t* empty = bars + kStages;      // [kStages]
  uint64_t* tfull = bars + 2 * kStages;  // [2]
  uint64_t* tempty = tfull + 2;          // [2]
  uint64_t* drain = tempty + 2;          // [1]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* aborted = reinterpret_cast<int*>(tmem_slot + 1);

  const int split = blockIdx.x, group = blockIdx.y, b = blockIdx.z;
  const int i0 = group * p.QN;
  const int nq = min(p.QN, p.Nq - i0);
  const int64_t t_last = p.q_pos0 + i0 + nq - 1;
  const int64_t nv_max = min(p.E, (t_last + 1) / p.m);
  const int64_t tiles = (nv_max + kTileM - 1) / kTileM;
  const int64_t tb = tiles * split / p.n_splits;
  const int64_t te = tiles * (split + 1) / p.n_splits;
  if (tb >= te) return;  // uniform over the CTA
  const int ntiles = (int)(te - tb);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- B operand: queries (generic-proxy writes, fenced to the async proxy below) ----------
  for (int idx = threadIdx.x; idx < p.ncols * 2; idx += kThreads) {
    const int r = idx >> 1, c = idx & 1;
    const int ql = r / CPQ, h = (r / NB) % H_I, blk = r % NB;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (ql < nq && c == blk) {
      const uint8_t* src =
          p.qi_codes + (((int64_t)b * p.Nq + i0 + ql) * H_I + h) * (NB * 16) + blk * 16;
      v = *reinterpret_cast<const uint4*>(src);
    }
    const int phys = r * kRowBytes + ((c ^ ((r >> 2) & 1)) << 4);  // 32-byte swizzle
    *reinterpret_cast<uint4*>(btile + phys) = v;
  }
  for (int r = threadIdx.x; r < p.ncols; r += kThreads) {
    const int ql = r / CPQ, h = (r / NB) % H_I, blk = r % NB;
    float s = 0.f;
    if (ql < nq)
      s = exp2_int((int)p.qi_scales[(((int64_t)b * p.Nq + i0 + ql) * H_I + h) * NB + blk] - 127);
    qscale[r] = s;
  }
  fence_proxy_async_smem();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *aborted = 0;
    fence_mbar_init();
    prefetch_tensormap(&kmap);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sfa_col = 2u * p.ncols, sfb_col = 2u * p.ncols + kSfCols;

  if (warp >= 2) {
    // scale factors = 1.0 everywhere in the two scale regions (all lanes of this quarter)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll
    for (int c = 0; c < 2 * kSfCols; c += 8) tmem_st8_fill(tmem + lane_base + sfa_col + c, 0x7F7F7F7Fu);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int issued = 0;
      for (int it = 0; it < ntiles; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (uint32_t)(it / kStages) & 1u;
        if (!mbar_wait(&empty[s], ph ^ 1u, p.status)) {
          *aborted = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kATileBytes);
        tma_load_3d(atiles + s * kATileBytes, &kmap, &full[s], 0, (int)((tb + it) * kTileM), b);
        ++issued;
      }
      if (*aborted) {  // let this CTA's own copies land before the CTA exits
        for (int it = max(0, issued - kStages); it < issued; ++it)
          mbar_wait(&full[it % kStages], (uint32_t)(it / kStages) & 1u, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_mxf4(kTileM, p.ncols);
      const uint64_t bdesc = smem_desc(smem_addr(btile), 16, 256, kSwizzle32B);
      for (int it = 0; it < ntiles; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (uint32_t)(it / kStages) & 1u;
        const int a = it & 1;
        const uint32_t aph = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(&tempty[a], aph ^ 1u, p.status) || !mbar_wait(&full[s], ph, p.status)) {
          *aborted = 1;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = smem_desc(smem_addr(atiles + s * kATileBytes), 16, 256, kSwizzle32B);
        umma_mxf4(tmem + (uint32_t)(a * p.ncols), adesc, bdesc, idesc, tmem + sfa_col,
                  tmem + sfb_col, 0u);
        umma_commit(&empty[s]);
        umma_commit(&tfull[a]);
      }
      umma_commit(drain);  // arrives once every MMA above has finished
      mbar_wait(drain, 0, p.status);
    }
  } else {
    // ---------------- epilogue: 4 warps, one tensor-memory lane quarter each ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    for (int it = 0; it < ntiles; ++it) {
      const int a = it & 1;
      const uint32_t aph = (uint32_t)(it >> 1) & 1u;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[a], aph, p.status) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) *aborted = 1;
        break;
      }
      tc_fence_after();
      const int64_t j = (tb + it) * kTileM + row;
      float sk[NB];
#pragma unroll
      for (int blk = 0; blk < NB; ++blk)
        sk[blk] = (j < p.E) ? exp2_int((int)p.ki_scales[((int64_t)b * p.E + j) * NB + blk] - 127)
                            : 0.f;
      for (int c0 = 0; c0 < p.ncols; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + (uint32_t)(a * p.ncols + c0), r);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 16; cc += CPQ) {
          const int ql = (c0 + cc) / CPQ;
          if (ql < nq) {
            float sc = 0.f;
#pragma unroll
            for (int h = 0; h < H_I; ++h) {
              float dot = 0.f;
#pragma unroll
              for (int blk = 0; blk < NB; ++blk)
                dot += (__uint_as_float(r[cc + h * NB + blk]) * qscale[c0 + cc + h * NB + blk]) *
                       sk[blk];
              sc += fmaxf(dot, 0.f);
            }
            sc += 0.0f;  // -0 -> +0
            const int64_t t = p.q_pos0 + i0 + ql;
            const int64_t nv = min(p.E, (t + 1) / p.m);
            if (j < nv) p.scores[((int64_t)b * p.Nq + i0 + ql) * p.E + j] = f32_to_bf16_bits(sc);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

template <int H_I, int NB>
cudaError_t launch_t(const CUtensorMap* kmap, const IdxParams& prm, const IndexerPlan& plan, int B,
                     cudaStream_t stream) {
  auto kern = indexer_kernel<H_I, NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)plan.n_splits, (unsigned)plan.n_groups, (unsigned)B);
  ProfScope prof(stream, "indexer_mxf4");
  kern<<<grid, kThreads, kSmemBytes, stream>>>(*kmap, prm);
  return cudaGetLastError();
}

int next_pow2_at_least32(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

IndexerPlan plan_indexer(int B, int Nq, int64_t E, int H_I, int d_I) {
  IndexerPlan pl{};
  const int cpq = H_I * (d_I / 32);
  if (Nq == 1) {
    pl.QN = 1;
    pl.ncols = 16;
  } else {
    pl.ncols = kMaxCols;
    pl.QN = kMaxCols / cpq;
  }
  pl.n_groups = (Nq + pl.QN - 1) / pl.QN;
  const int64_t tiles = (E + kTileM - 1) / kTileM;
  const int64_t units = (int64_t)B * pl.n_groups;
  const int64_t target = (int64_t)kNumSMs * 4;
  int64_t splits = (target + units - 1) / units;
  if (splits > tiles) splits = tiles;
  if (splits < 1) splits = 1;
  pl.n_splits = (int)splits;
  pl.tmem_cols = next_pow2_at_least32(2 * pl.ncols + 2 * kSfCols);
  return pl;
}

cudaError_t launch_indexer(const CUtensorMap* kmap, const uint8_t* qi_codes,
                           const uint8_t* qi_scales, const uint8_t* ki_scales, uint16_t* scores,
                           int B, int Nq, int64_t q_pos0, int64_t E, int m, int H_I, int d_I,
                           const IndexerPlan& plan, uint32_t* status, cudaStream_t stream) {
  IdxParams prm;
  prm.qi_codes = qi_codes;
  prm.qi_scales = qi_scales;
  prm.ki_scales = ki_scales;
  prm.scores = scores;
  prm.q_pos0 = q_pos0;
  prm.E = E;
  prm.Nq = Nq;
  prm.m = m;
  prm.QN = plan.QN;
  prm.ncols = plan.ncols;
  prm.n_splits = plan.n_splits;
  prm.tmem_cols = plan.tmem_cols;
  prm.status = status;
  const int NB = d_I / 32;
#define CSA_IDX_CASE(HH, NN) \
  if (H_I == HH && NB == NN) return launch_t<HH, NN>(kmap, prm, plan, B, stream);
  CSA_IDX_CASE(1, 1) CSA_IDX_CASE(2, 1) CSA_IDX_CASE(4, 1) CSA_IDX_CASE(8, 1)
  CSA_IDX_CASE(1, 2) CSA_IDX_CASE(2, 2) CSA_IDX_CASE(4, 2) CSA_IDX_CASE(8, 2)
#undef CSA_IDX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace csa
