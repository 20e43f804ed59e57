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
// (t % m == m - 1) pools the block's m rows (the ring's, and token t's straight from the
// inputs) with the softmax of their logits into entry t / m of its page: fp32 sums over 16
// token groups of 64 channel pairs, each thread keeping eight rows in flight, bf16 entries. A
// CSA layer also pools the index-key rows and converts the key to MX FP4 with the arithmetic
// of csa_compress_index_keys.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kThreads = 1024;
constexpr int kGroups = 16;                // token groups: group g pools the tokens i = g mod 16
constexpr int kPairs = kThreads / kGroups; // 64 channel pairs: one 32-bit word of a d = 128 row
constexpr int kBatch = 8;                  // rows in flight per thread

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

// d = 128 (the paged path's head dim): a row is 64 32-bit words of two bf16 channels.
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendParams p) {
  __shared__ float w_s[kRingTokens];
  __shared__ float red[2];
  __shared__ float4 part[kGroups][kPairs];  // (k lo, k hi, v lo, v hi) partial sums per group
  pdl_wait();  // the ring and pages may still be read by the previous step's kernels
  pdl_trigger();
  const PagedLayout& L = p.L;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int m = L.m;
  const int64_t t = p.t;
  const int slot = (int)(t & (kRingTokens - 1));
  const int64_t rb = (int64_t)b * kRingTokens;
  const uint32_t* rk = reinterpret_cast<const uint32_t*>(L.ring_k);
  const uint32_t* rv = reinterpret_cast<const uint32_t*>(L.ring_v);
  const uint32_t* kn = reinterpret_cast<const uint32_t*>(p.k_new) + (int64_t)b * kPairs;
  const uint32_t* vn = reinterpret_cast<const uint32_t*>(p.v_new) + (int64_t)b * kPairs;
  // ---- the new token into the state cache ----
  if (tid < kPairs) {
    reinterpret_cast<uint32_t*>(L.ring_k)[(rb + slot) * kPairs + tid] = kn[tid];
    reinterpret_cast<uint32_t*>(L.ring_v)[(rb + slot) * kPairs + tid] = vn[tid];
  }
  if (tid == 0) L.ring_logits[rb + slot] = p.logit_new[b];
  if (L.ring_xi && p.xi_new && tid < L.d_I)
    L.ring_xi[(rb + slot) * L.d_I + tid] = p.xi_new[(int64_t)b * L.d_I + tid];
  if ((t % m) != m - 1) return;  // no block closes (uniform over the CTA)

  // ---- pool block j = t / m: rows t - m + 1 .. t - 1 from the ring, row t from the inputs ----
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
  const int g = tid / kPairs, c = tid % kPairs;
  auto row_k = [&](int i) -> uint32_t {
    return i == m - 1 ? kn[c] : rk[(rb + ((t0 + i) & (kRingTokens - 1))) * kPairs + c];
  };
  auto row_v = [&](int i) -> uint32_t {
    return i == m - 1 ? vn[c] : rv[(rb + ((t0 + i) & (kRingTokens - 1))) * kPairs + c];
  };
  // the first batch of this thread's rows is requested before the weights are reduced
  uint32_t kb[kBatch], vb[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int i = g + kGroups * u;
    if (i < m) {
      kb[u] = row_k(i);
      vb[u] = row_v(i);
    }
  }
  // softmax weights of the block's logits (m <= 128), warp 0
  for (int i = tid; i < m; i += kThreads)
    w_s[i] = i == m - 1 ? p.logit_new[b] : L.ring_logits[rb + ((t0 + i) & (kRingTokens - 1))];
  __syncthreads();
  if (tid < 32) {
    float mx = -INFINITY;
    for (int i = tid; i < m; i += 32) mx = fmaxf(mx, w_s[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float ex[kRingTokens / 32];
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < kRingTokens / 32; ++u) {
      const int i = tid + 32 * u;
      ex[u] = i < m ? expf(w_s[i] - mx) : 0.f;
      sum += ex[u];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kRingTokens / 32; ++u)
      if (tid + 32 * u < m) w_s[tid + 32 * u] = ex[u];
    if (tid == 0) red[0] = 1.f / sum;
  }
  __syncthreads();
  const float inv = red[0];
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (int base = 0; base < m; base += kGroups * kBatch) {
    if (base > 0) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = base + g + kGroups * u;
        if (i < m) {
          kb[u] = row_k(i);
          vb[u] = row_v(i);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = base + g + kGroups * u;
      if (i < m) {
        const float pw = w_s[i] * inv;
        a0 = fmaf(pw, __uint_as_float(kb[u] << 16), a0);
        a1 = fmaf(pw, __uint_as_float(kb[u] & 0xFFFF0000u), a1);
        a2 = fmaf(pw, __uint_as_float(vb[u] << 16), a2);
        a3 = fmaf(pw, __uint_as_float(vb[u] & 0xFFFF0000u), a3);
      }
    }
  }
  part[g][c] = make_float4(a0, a1, a2, a3);
  __syncthreads();
  if (g == 0) {
    float4 s4 = part[0][c];
#pragma unroll
    for (int q = 1; q < kGroups; ++q) {
      const float4 o = part[q][c];
      s4.x += o.x;
      s4.y += o.y;
      s4.z += o.z;
      s4.w += o.w;
    }
    reinterpret_cast<uint32_t*>(L.k_pool)[dst * kPairs + c] = pack_bf16x2(s4.x, s4.y);
    reinterpret_cast<uint32_t*>(L.v_pool)[dst * kPairs + c] = pack_bf16x2(s4.z, s4.w);
  }
  if (!L.ring_xi || !L.ki_codes_pool || !p.xi_new) return;
  // ---- the indexer's key of the entry: pooled, bf16, MX FP4 (one element per thread), with
  // the arithmetic of csa_compress_index_keys (weights e_i / sum in token order) ----
  const int dI = L.d_I;  // 32, 64 or 128 <= kThreads
  uint32_t bits = 0;
  if (tid < dI) {
    float ax = 0.f;
    for (int i = 0; i < m; ++i) {
      const uint16_t x = i == m - 1 ? p.xi_new[(int64_t)b * dI + tid]
                                    : L.ring_xi[(rb + ((t0 + i) & (kRingTokens - 1))) * dI + tid];
      ax = fmaf(w_s[i] * inv, bf16_bits_to_f32(x), ax);
    }
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
  if (L.d != 2 * kPairs || L.m > kRingTokens / 2) return cudaErrorInvalidValue;
  AppendParams prm{L, k_new, v_new, logit_new, xi_new, t, status};
  ProfScope prof(stream, "paged_append");
  return launch_ex(append_kernel, dim3((unsigned)B), dim3(kThreads), 0, stream, 1, prm);
}

}  // namespace csa
