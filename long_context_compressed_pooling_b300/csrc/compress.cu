// Block pooling of raw K/V into compressed entries (CSA m = 4, HCA m = 128).
//
// Lighthouse "deep deepseek v4 release" 八.3: every m consecutive KV tokens are merged into
// one compressed entry. Pooling operator (not printed on the pages; the workload definition
// fixes it): p_i = softmax_i(w[jm+i]) over the block's per-token logits, entry = sum_i p_i row_i,
// the same weights for K and V.
//
// HBM-bound streaming kernel: every raw byte is read once with 128-bit loads, every entry
// byte written once. One thread owns 8 channels (16 bytes) of one entry for both K and V,
// so a warp reads 512 contiguous bytes per token row pair.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

// grid-stride over (b, entry, 16-byte chunk); CH = d / 8 chunks per row.
template <int CH>
__global__ void __launch_bounds__(256) compress_kernel(const uint16_t* __restrict__ k_raw,
                                                       const uint16_t* __restrict__ v_raw,
                                                       const float* __restrict__ logits,
                                                       uint16_t* __restrict__ k_cmp,
                                                       uint16_t* __restrict__ v_cmp, int B,
                                                       int64_t N, int m, int64_t j_begin,
                                                       int64_t n_entries) {
  constexpr int D = CH * 8;
  // wait before letting the successor start: a successor that reads entries this launch does
  // not write, before its own wait, then also sees every earlier kernel complete
  pdl_wait();
  pdl_trigger();
  const int64_t E = N / m;
  const int64_t total = (int64_t)B * n_entries * CH;
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < total;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(w % CH);
    const int64_t e = (w / CH) % n_entries;
    const int64_t b = w / ((int64_t)CH * n_entries);
    const int64_t j = j_begin + e;
    const int64_t tok0 = b * N + j * m;
    const float* wl = logits + tok0;

    const uint16_t* kp = k_raw + tok0 * D + c * 8;
    const uint16_t* vp = v_raw + tok0 * D + c * 8;
    // the first four rows are requested before the logits' maximum is known
    uint4 kv[4], vv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (u < m) {
        kv[u] = ldg_stream(kp + (int64_t)u * D);
        vv[u] = ldg_stream(vp + (int64_t)u * D);
      }
    float mx = -INFINITY;
    for (int i = 0; i < m; ++i) mx = fmaxf(mx, __ldg(wl + i));

    float acc_k[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float acc_v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float sum = 0.f;
    int i = 0;
    for (; i + 4 <= m; i += 4) {
      if (i > 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          kv[u] = ldg_stream(kp + (int64_t)(i + u) * D);
          vv[u] = ldg_stream(vp + (int64_t)(i + u) * D);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float p = expf(__ldg(wl + i + u) - mx);
        sum += p;
        acc8(acc_k, kv[u], p);
        acc8(acc_v, vv[u], p);
      }
    }
    if (m < 4) {  // blocks shorter than four rows: all of them are already loaded
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (u < m) {
          const float p = expf(__ldg(wl + u) - mx);
          sum += p;
          acc8(acc_k, kv[u], p);
          acc8(acc_v, vv[u], p);
        }
    } else {
      for (; i < m; ++i) {  // ragged tail of m >= 4 (not a multiple of 4)
        const float p = expf(__ldg(wl + i) - mx);
        sum += p;
        acc8(acc_k, ldg_stream(kp + (int64_t)i * D), p);
        acc8(acc_v, ldg_stream(vp + (int64_t)i * D), p);
      }
    }
    const float inv = 1.0f / sum;
    const int64_t o = (b * E + j) * D + c * 8;
    *reinterpret_cast<uint4*>(k_cmp + o) = pack8(acc_k, inv);
    *reinterpret_cast<uint4*>(v_cmp + o) = pack8(acc_v, inv);
  }
}

// Large blocks (m >= 32): one CTA per entry. The block's softmax weights are computed once into
// shared memory; thread (slice, chunk) accumulates the tokens slice, slice+TS, ... of 16-byte
// channel chunk `chunk` for K and V, so all of a thread's loads are independent and in flight
// together; the TS partial sums are then reduced through shared memory.
template <int CH>
__global__ void __launch_bounds__(256) compress_large_kernel(const uint16_t* __restrict__ k_raw,
                                                             const uint16_t* __restrict__ v_raw,
                                                             const float* __restrict__ logits,
                                                             uint16_t* __restrict__ k_cmp,
                                                             uint16_t* __restrict__ v_cmp, int B,
                                                             int64_t N, int m, int64_t j_begin,
                                                             int64_t n_entries) {
  constexpr int D = CH * 8;
  constexpr int TS = 256 / CH;  // token slices
  __shared__ float wexp[256];
  __shared__ float red[2];
  __shared__ float part[2][TS][CH * 8 + 1];
  const int tid = threadIdx.x;
  const int c = tid % CH, ts = tid / CH;
  const int64_t E = N / m;
  pdl_wait();  // before the trigger, as in compress_kernel
  pdl_trigger();
  for (int64_t w = blockIdx.x; w < (int64_t)B * n_entries; w += gridDim.x) {
    const int64_t b = w / n_entries, j = j_begin + w % n_entries;
    const int64_t tok0 = b * N + j * m;
    // The first kBatch of this thread's tokens (ts, ts + TS, ...) are loaded before the softmax
    // weights are formed: their loads do not depend on the weights and overlap the reductions.
    constexpr int kBatch = 8;
    const uint16_t* kp = k_raw + tok0 * D + c * 8;
    const uint16_t* vp = v_raw + tok0 * D + c * 8;
    uint4 kv[kBatch], vv[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = ts + u * TS;
      if (i < m) {
        kv[u] = ldg_stream(kp + (int64_t)i * D);
        vv[u] = ldg_stream(vp + (int64_t)i * D);
      }
    }
    // softmax weights of the block (m <= 256)
    const float x = tid < m ? __ldg(logits + tok0 + tid) : -INFINITY;
    float mx = x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((tid & 31) == 0) wexp[tid >> 5] = mx;  // per-warp maxima (scratch)
    __syncthreads();
    if (tid == 0) {
      float M = wexp[0];
      for (int q = 1; q < 8; ++q) M = fmaxf(M, wexp[q]);
      red[0] = M;
    }
    __syncthreads();
    const float e = tid < m ? expf(x - red[0]) : 0.f;
    float sm = e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, o);
    __syncthreads();
    if ((tid & 31) == 0) wexp[tid >> 5] = sm;
    __syncthreads();
    if (tid == 0) {
      float S = 0.f;
      for (int q = 0; q < 8; ++q) S += wexp[q];
      red[1] = S;
    }
    __syncthreads();
    wexp[tid] = e;
    __syncthreads();

    float acc_k[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float acc_v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i = ts + u * TS;
      if (i < m) {
        acc8(acc_k, kv[u], wexp[i]);
        acc8(acc_v, vv[u], wexp[i]);
      }
    }
    for (int i = ts + kBatch * TS; i < m; i += TS) {  // blocks longer than kBatch * TS tokens
      acc8(acc_k, ldg_stream(kp + (int64_t)i * D), wexp[i]);
      acc8(acc_v, ldg_stream(vp + (int64_t)i * D), wexp[i]);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      part[0][ts][c * 8 + q] = acc_k[q];
      part[1][ts][c * 8 + q] = acc_v[q];
    }
    __syncthreads();
    // 2 * D outputs; thread tid reduces output channel tid of K (tid < D) or V (tid >= D)
    const float inv = 1.0f / red[1];
    for (int o = tid; o < 2 * D; o += 256) {
      const int kv = o / D, ch = o % D;
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < TS; ++q) s += part[kv][q][ch];
      uint16_t* dst = (kv == 0 ? k_cmp : v_cmp) + (b * E + j) * D + ch;
      *dst = f32_to_bf16_bits(s * inv);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------------
// The Lightning Indexer's own compressed keys (Lighthouse 八.7 lists them beside the CSA / HCA
// entries; 9fzt.com item 4 runs the indexer's QK path in FP4): per-token index-key rows are
// pooled with the same block pooling, rounded to bf16, and converted to MX FP4 (OCP
// Microscaling Formats v1.0, section 6.3: block scale X = 2^(floor(log2 max|v|) - 2), elements
// v / X rounded to nearest-even on the E2M1 grid and clamped to 6; an all-zero block takes the
// smallest scale byte 0). One warp per row: lane l holds elements [EPL l, EPL l + EPL) of a
// d = 32 EPL row, so a 32-element block spans 32 / EPL lanes.
// ---------------------------------------------------------------------------------------------

// E2M1 code (3 magnitude bits) of |y|: the nearest grid value, ties to the even code. The grid
// midpoints are 0.25 0.75 1.25 1.75 2.5 3.5 5; at a midpoint the even neighbour wins, so the
// comparison is strict where the lower neighbour is even and inclusive where the upper one is.
CSA_DEV uint32_t e2m1_magnitude_code(float a) {
  return (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
         (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) + (uint32_t)(a > 5.0f);
}

// Converts this lane's EPL bf16 values (bit patterns) of a row to E2M1 codes (low nibbles,
// element order) and returns the block's UE8M0 scale byte (valid in every lane of the block).
template <int EPL>
CSA_DEV uint32_t mx_encode(const uint32_t (&bits)[EPL], uint32_t (&code)[EPL]) {
  constexpr int LPB = 32 / EPL;  // lanes per 32-element block
  uint32_t amax = 0;  // |v| as fp32 bits: order-preserving for non-negative values
#pragma unroll
  for (int e = 0; e < EPL; ++e) amax = max(amax, (bits[e] << 16) & 0x7FFFFFFFu);
#pragma unroll
  for (int o = 1; o < LPB; o <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // floor(log2 amax) - 2, clamped to the UE8M0 range; a zero (or bf16 subnormal) maximum gives
  // the smallest scale
  const int ef = (int)(amax >> 23);
  const int xe = ef == 0 ? -127 : max(ef - 129, -127);
  const float inv_x = __int_as_float((127 - xe) << 23);  // 2^-xe, exact
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const float v = __uint_as_float(bits[e] << 16);
    code[e] = e2m1_magnitude_code(fabsf(v) * inv_x) | ((bits[e] >> 12) & 0x8u);
  }
  return (uint32_t)(xe + 127);
}

// Writes one row's codes (d / 2 bytes) and scales (d / 32 bytes).
template <int EPL>
CSA_DEV void mx_store(const uint32_t (&code)[EPL], uint32_t scale, uint8_t* codes_row,
                      uint8_t* scales_row, int lane) {
  constexpr int LPB = 32 / EPL;
  if constexpr (EPL == 1) {
    const uint32_t hi = __shfl_down_sync(0xffffffffu, code[0], 1);
    if ((lane & 1) == 0) codes_row[lane >> 1] = (uint8_t)(code[0] | (hi << 4));
  } else if constexpr (EPL == 2) {
    codes_row[lane] = (uint8_t)(code[0] | (code[1] << 4));
  } else {
    *reinterpret_cast<uint16_t*>(codes_row + 2 * lane) =
        (uint16_t)(code[0] | (code[1] << 4) | (code[2] << 8) | (code[3] << 12));
  }
  if (lane % LPB == 0) scales_row[lane / LPB] = (uint8_t)scale;
}

template <int EPL>
CSA_DEV void load_row(const uint16_t* row, int lane, uint32_t (&bits)[EPL]) {
  if constexpr (EPL == 1) {
    bits[0] = row[lane];
  } else if constexpr (EPL == 2) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(row + 2 * lane);
    bits[0] = u & 0xFFFFu;
    bits[1] = u >> 16;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(row + 4 * lane);
    bits[0] = u.x & 0xFFFFu;
    bits[1] = u.x >> 16;
    bits[2] = u.y & 0xFFFFu;
    bits[3] = u.y >> 16;
  }
}

// Index keys of entries [j_begin, j_begin + n_entries) of every sequence; m <= 32 (one lane per
// token of the block holds its logit).
template <int EPL>
__global__ void __launch_bounds__(256) index_keys_kernel(const uint16_t* __restrict__ xi_raw,
                                                         const float* __restrict__ logits,
                                                         uint8_t* __restrict__ ki_codes,
                                                         uint8_t* __restrict__ ki_scales, int B,
                                                         int64_t N, int m, int64_t j_begin,
                                                         int64_t n_entries) {
  constexpr int D = 32 * EPL;
  pdl_wait();  // before the trigger, as in compress_kernel
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t E = N / m;
  const int64_t total = (int64_t)B * n_entries;
  for (int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); w < total;
       w += (int64_t)gridDim.x * 8) {
    const int64_t b = w / n_entries, j = j_begin + w % n_entries;
    const int64_t t0 = b * N + j * m;  // first token of the block
    const float lg = lane < m ? logits[t0 + lane] : -INFINITY;
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float mx = lg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ex = lane < m ? expf(lg - mx) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = 1.f / sum;
    for (int i0 = 0; i0 < m; i0 += 4) {
      uint32_t rb[4][EPL];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i0 + u < m) load_row<EPL>(xi_raw + (t0 + i0 + u) * D, lane, rb[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float pw = __shfl_sync(0xffffffffu, ex, (i0 + u) & 31) * inv;
        if (i0 + u < m) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pw, __uint_as_float(rb[u][e] << 16), acc[e]);
        }
      }
    }
    uint32_t bits[EPL], code[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      bits[e] = f32_to_bf16_bits(acc[e]);
      if (bits[e] == 0x8000u) bits[e] = 0u;  // a pooled zero is +0
    }
    const uint32_t scale = mx_encode<EPL>(bits, code);
    const int64_t row = b * E + j;
    mx_store<EPL>(code, scale, ki_codes + row * (D / 2), ki_scales + row * (D / 32), lane);
  }
}

// MX FP4 conversion of bf16 rows (the index queries), one warp per row.
template <int EPL>
__global__ void __launch_bounds__(256) mxfp4_quantize_kernel(const uint16_t* __restrict__ x,
                                                             int64_t rows,
                                                             uint8_t* __restrict__ codes,
                                                             uint8_t* __restrict__ scales) {
  constexpr int D = 32 * EPL;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  for (int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); r < rows;
       r += (int64_t)gridDim.x * 8) {
    uint32_t bits[EPL], code[EPL];
    load_row<EPL>(x + r * D, lane, bits);
    const uint32_t scale = mx_encode<EPL>(bits, code);
    mx_store<EPL>(code, scale, codes + r * (D / 2), scales + r * (D / 32), lane);
  }
}

}  // namespace

cudaError_t launch_compress(const uint16_t* k_raw, const uint16_t* v_raw, const float* logits,
                            int B, int64_t N, int d, int m, int64_t j_begin, int64_t n_entries,
                            uint16_t* k_cmp, uint16_t* v_cmp, cudaStream_t stream) {
  if (n_entries <= 0 || B <= 0) return cudaSuccess;
  const int ch = d / 8;
  if (m >= 32 && ch <= 32) {
    int64_t blocks = (int64_t)B * n_entries;
    const int64_t cap = (int64_t)kNumSMs * 8;
    if (blocks > cap) blocks = cap;
    ProfScope prof(stream, "compress");
    cudaError_t e = cudaSuccess;
    switch (ch) {
      case 8:
        e = launch_ex(compress_large_kernel<8>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                      k_raw, v_raw, logits, k_cmp, v_cmp, B, N, m, j_begin, n_entries);
        break;
      case 16:
        e = launch_ex(compress_large_kernel<16>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                      k_raw, v_raw, logits, k_cmp, v_cmp, B, N, m, j_begin, n_entries);
        break;
      case 32:
        e = launch_ex(compress_large_kernel<32>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                      k_raw, v_raw, logits, k_cmp, v_cmp, B, N, m, j_begin, n_entries);
        break;
      default:
        return cudaErrorInvalidValue;
    }
    return e;
  }
  const int64_t total = (int64_t)B * n_entries * ch;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)kNumSMs * 8;  // 8 resident 256-thread CTAs per SM
  if (blocks > cap) blocks = cap;
  ProfScope prof(stream, "compress");
  cudaError_t e = cudaSuccess;
  switch (ch) {
    case 8:
      e = launch_ex(compress_kernel<8>, dim3((unsigned)blocks), dim3(threads), 0, stream, 1,
                    k_raw, v_raw, logits, k_cmp, v_cmp, B, N, m, j_begin, n_entries);
      break;
    case 16:
      e = launch_ex(compress_kernel<16>, dim3((unsigned)blocks), dim3(threads), 0, stream, 1,
                    k_raw, v_raw, logits, k_cmp, v_cmp, B, N, m, j_begin, n_entries);
      break;
    case 32:
      e = launch_ex(compress_kernel<32>, dim3((unsigned)blocks), dim3(threads), 0, stream, 1,
                    k_raw, v_raw, logits, k_cmp, v_cmp, B, N, m, j_begin, n_entries);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return e;
}

cudaError_t launch_index_keys(const uint16_t* xi_raw, const float* logits, int B, int64_t N, int d_I,
                              int m, int64_t j_begin, int64_t n_entries, uint8_t* ki_codes,
                              uint8_t* ki_scales, cudaStream_t stream) {
  if (n_entries <= 0 || B <= 0) return cudaSuccess;
  int64_t blocks = ((int64_t)B * n_entries + 7) / 8;
  const int64_t cap = (int64_t)kNumSMs * 8;
  if (blocks > cap) blocks = cap;
  ProfScope prof(stream, "index_keys");
  switch (d_I) {
    case 32:
      return launch_ex(index_keys_kernel<1>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                       xi_raw, logits, ki_codes, ki_scales, B, N, m, j_begin, n_entries);
    case 64:
      return launch_ex(index_keys_kernel<2>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                       xi_raw, logits, ki_codes, ki_scales, B, N, m, j_begin, n_entries);
    case 128:
      return launch_ex(index_keys_kernel<4>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                       xi_raw, logits, ki_codes, ki_scales, B, N, m, j_begin, n_entries);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_mxfp4_quantize(const uint16_t* x, int64_t rows, int d, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = (int64_t)kNumSMs * 8;
  if (blocks > cap) blocks = cap;
  ProfScope prof(stream, "mxfp4_quantize");
  switch (d) {
    case 32:
      return launch_ex(mxfp4_quantize_kernel<1>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                       x, rows, codes, scales);
    case 64:
      return launch_ex(mxfp4_quantize_kernel<2>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                       x, rows, codes, scales);
    case 128:
      return launch_ex(mxfp4_quantize_kernel<4>, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                       x, rows, codes, scales);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace csa
