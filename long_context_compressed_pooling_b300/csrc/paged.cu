// Paged heterogeneous KV cache: appending one decoded token and compressing the blocks it
// completes (Lighthouse "deep deepseek v4 release" 八.7: a state cache for the sliding window and
// the not yet compressed tail, a classical cache for the compressed entries, cache blocks
// aligned to lcm(m, m') tokens).
//
// Layout (one layer):
//   classical cache  pools of pages; a page holds the entries of kPageTokens = 4096 consecutive
//                    tokens of one sequence (4096 / m entries: 1024 CSA entries and their index
//                    keys, or 32 HCA entries); block_table[b][i] names the page of tokens
//                    [4096 i, 4096 (i + 1)) of sequence b. 4096 is a multiple of lcm(4, 128), so
//                    every block of m tokens lies in one page.
//   state cache      a ring of the last kRingTokens = 256 raw tokens per sequence (K, V rows,
//                    pooling logits, index-key rows): the window (W <= 128) and the longest
//                    pending tail (m - 1 <= 127 tokens) always fit.
//
// One CTA per sequence: it writes token t into ring slot t % 256, and when t closes a block
// (t % m == m - 1) pools the block's m ring rows with the softmax of their logits into entry
// t / m of its page, with the same arithmetic as the flat compressor (fp32 sums, bf16 entries);
// a CSA layer also pools the index-key rows and converts the key to MX FP4 as
// csa_compress_index_keys does.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kThreads = 128;

struct AppendParams {
  PagedLayout L;
  const uint16_t* k_new;     // [B, d]
  const uint16_t* v_new;     // [B, d]
  const float* logit_new;    // [B]
  const uint16_t* xi_new;    // [B, d_I] (CSA with index keys) or null
  int64_t t;                 // position of the appended token
  uint32_t* status;
};

// E2M1 code of |y| (nearest, ties to even), as in the compressor's index-key path.
CSA_DEV uint32_t e2m1_code(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
         (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
}

__global__ void __launch_bounds__(kThreads) append_kernel(const AppendParams p) {
  __shared__ float w_s[kRingTokens];
  __shared__ float red[2];
  pdl_wait();  // the ring and pages may still be read by the previous step's kernels
  pdl_trigger();
  const PagedLayout& L = p.L;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int d = L.d, m = L.m;
  const int64_t t = p.t;
  const int slot = (int)(t % kRingTokens);
  const int64_t rb = (int64_t)b * kRingTokens;
  // ---- the new token into the state cache ----
  for (int c = tid; c < d; c += kThreads) {
    L.ring_k[(rb + slot) * d + c] = p.k_new[(int64_t)b * d + c];
    L.ring_v[(rb + slot) * d + c] = p.v_new[(int64_t)b * d + c];
  }
  if (tid == 0) L.ring_logits[rb + slot] = p.logit_new[b];
  if (L.ring_xi && p.xi_new)
    for (int c = tid; c < L.d_I; c += kThreads)
      L.ring_xi[(rb + slot) * L.d_I + c] = p.xi_new[(int64_t)b * L.d_I + c];
  if ((t % m) != m - 1) return;  // no block closes (uniform over the CTA)
  __syncthreads();               // the ring rows of the block, the new one included

  // ---- pool block j = t / m ----
  const int64_t j = t / m;
  const int64_t t0 = t - (m - 1);
  const int64_t blk = (j * m) / kPageTokens;
  const int page = blk < L.max_blocks ? L.block_table[(int64_t)b * L.max_blocks + blk] : -1;
  if (page < 0 || page >= L.n_pages) {
    if (tid == 0) atomicOr(p.status, kFlagBadIndex);  // unmapped page: nothing is written
    return;
  }
  const int per_page = kPageTokens / m;
  const int64_t dst = (int64_t)page * per_page + (j % per_page);  // entry row in the pool
  // softmax weights of the block's logits (m <= 128)
  if (tid < 32) {
    float mx = -INFINITY;
    for (int i = tid; i < m; i += 32) {
      const float lg = L.ring_logits[rb + (t0 + i) % kRingTokens];
      w_s[i] = lg;
      mx = fmaxf(mx, lg);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int i = tid; i < m; i += 32) {
      const float e = expf(w_s[i] - mx);
      w_s[i] = e;
      sum += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (tid == 0) red[0] = 1.f / sum;
  }
  __syncthreads();
  const float inv = red[0];
  for (int c = tid; c < d; c += kThreads) {
    float ak = 0.f, av = 0.f;
    for (int i = 0; i < m; ++i) {
      const int64_t r = (rb + (t0 + i) % kRingTokens) * d + c;
      const float pw = w_s[i] * inv;
      ak = fmaf(pw, bf16_bits_to_f32(L.ring_k[r]), ak);
      av = fmaf(pw, bf16_bits_to_f32(L.ring_v[r]), av);
    }
    L.k_pool[dst * d + c] = f32_to_bf16_bits(ak);
    L.v_pool[dst * d + c] = f32_to_bf16_bits(av);
  }
  if (!L.ring_xi || !L.ki_codes_pool) return;
  // ---- the indexer's key of the entry: pooled, bf16, MX FP4 (one element per thread) ----
  const int dI = L.d_I;  // 32, 64 or 128 <= kThreads
  uint32_t bits = 0;
  if (tid < dI) {
    float ax = 0.f;
    for (int i = 0; i < m; ++i)
      ax = fmaf(w_s[i] * inv,
                bf16_bits_to_f32(L.ring_xi[(rb + (t0 + i) % kRingTokens) * dI + tid]), ax);
    bits = f32_to_bf16_bits(ax);
    if (bits == 0x8000u) bits = 0u;  // a pooled zero is +0
  }
  // block maximum: each warp is one 32-element block
  uint32_t amax = (bits << 16) & 0x7FFFFFFFu;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int ef = (int)(amax >> 23);
  const int xe = ef == 0 ? -127 : max(ef - 129, -127);
  const float inv_x = __int_as_float((127 - xe) << 23);
  const uint32_t code =
      e2m1_code(fabsf(__uint_as_float(bits << 16)) * inv_x) | ((bits >> 12) & 0x8u);
  const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);
  if (tid < dI) {
    if ((tid & 1) == 0) L.ki_codes_pool[dst * (dI / 2) + tid / 2] = (uint8_t)(code | (hi << 4));
    if ((tid & 31) == 0) L.ki_scales_pool[dst * (dI / 32) + tid / 32] = (uint8_t)(xe + 127);
  }
}

}  // namespace

cudaError_t launch_paged_append(const PagedLayout& L, int B, const uint16_t* k_new,
                                const uint16_t* v_new, const float* logit_new,
                                const uint16_t* xi_new, int64_t t, uint32_t* status,
                                cudaStream_t stream) {
  if (B <= 0) return cudaSuccess;
  AppendParams prm{L, k_new, v_new, logit_new, xi_new, t, status};
  ProfScope prof(stream, "paged_append");
  return launch_ex(append_kernel, dim3((unsigned)B), dim3(kThreads), 0, stream, 1, prm);
}

}  // namespace csa
