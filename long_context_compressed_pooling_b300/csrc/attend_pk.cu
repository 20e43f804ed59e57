// CSA sparse and HCA dense attention for head dim 64 on the 5th-generation tensor cores
// (tcgen05), prefill: several query tokens packed into the M = 64 rows of one CTA.
//
// Lighthouse "deep deepseek v4 release" 八.3: CSA attends to the top-k selected compressed
// entries plus a sliding-window branch of raw tokens; HCA attends densely to every compressed
// entry plus the same window. One softmax spans a query's entries and window tokens; logits are
// q.k (the 1/sqrt(d) is folded into q).
//
// With few heads (the small configuration has 8 heads of 64) one token fills only H of the
// MMA's 64 rows, so a CTA takes G = 64 / Hp consecutive query tokens of one sequence (Hp = H
// rounded up to a power of two): row r = g * Hp + h is head h of token g. The tokens share one
// key list and every row masks the keys that are not its own:
//   sparse (CSA): slot g * k + i holds entry topk_idx[token g][i] (i < its count), valid for the
//                 rows of token g only;
//   dense (HCA):  entry j (j below the last token's visible count), valid for the rows of token g
//                 while j < visible(t_g);
//   window:       raw tokens [t_first - W + 1, t_last], valid for token g inside its own window.
// The loaders write a tag per key (owner token, entry index or window offset) next to the tiles;
// the softmax turns tag and row into validity. Then, per 128-key chunk:
//   S[64 rows, 128 keys] = Q[64, 64 d] . K_chunk^T    (4 MMAs, K = 16 each)
//   O[64 rows, 64 d]    += P[64, 128 keys] . V_chunk  (8 MMAs; keys 0-63 and 64-127 into two
//                                                     accumulators, one per softmax key half)
// with S double-buffered in tensor memory, 4 K/V stages of 32 KB, the same warp roles as the
// d = 128 kernel (8 softmax warps, 8 loader warps, one MMA warp) and bounded waits throughout.
// Decode (one query per sequence) keeps the split-K mma.sync kernel of attend.cu.
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kD = 64;             // head dim
constexpr int kM = 64;             // rows per CTA (MMA M)
constexpr int kKC = 128;           // keys per chunk (N of QK^T, K of PV)
constexpr int kHalf = kKC / 2;     // keys per softmax warp (and per O accumulator)
constexpr int kStages = 4;         // K/V stages
constexpr int kSoftmaxWarps = 8;   // warps 0-7: lane quarter w % 4, key half w / 4
constexpr int kLoadWarp0 = 8;      // warps 8-15
constexpr int kLoadWarps = 8;
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kMmaWarp = 16;
constexpr int kThreads = 544;
constexpr int kSetupThreads = 32 * (kSoftmaxWarps + 1);  // softmax warps + MMA warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;    // O accumulators: key half 0 at [256, 320), half 1 at [320, 384)
constexpr int kQBytes = kM * kD * 2;        // 8 KB: one 128-byte swizzle atom of 64 rows
constexpr int kTileBytes = kKC * kD * 2;    // 16 KB (one K or V tile)
constexpr int kPBytes = kM * kKC * 2;       // 16 KB
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kNumBars = 16;
constexpr int kMaxG = 64;                   // tokens per CTA (H = 1)
// key tags: -1 none; owner token g (sparse entries); kTagEntry | j (dense entry j); kTagWin | o
// (window token wlo + o)
constexpr int32_t kTagEntry = 0x40000000;
constexpr int32_t kTagWin = 0x20000000;
constexpr int32_t kTagLow = 0x1FFFFFFF;
constexpr size_t kSmemBytes = 1024 + kQBytes + (size_t)kStages * 2 * kTileBytes + kPBytes +
                              (size_t)kStages * kKC * 4 /*tags*/ + kMaxG * 4 * 4 /*per token*/ +
                              kNumBars * 8 + 16 + 2 * kM * 2 * 4;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct PkParams {
  const uint16_t* q;
  const uint16_t* k_cmp;
  const uint16_t* v_cmp;
  const int32_t* topk_idx;
  const int32_t* topk_cnt;
  const uint16_t* k_raw;
  const uint16_t* v_raw;
  uint16_t* out;
  float* lse;
  int64_t E, N, q_pos0;
  int k, m, W, Nq, H, Hp, G, groups;  // groups: query groups per sequence
  int sparse;
  uint32_t* status;
};

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled K-major tile of 64
// bf16 columns (one atom): chunk index XOR (row mod 8).
CSA_DEV uint32_t sw64(int r, int c) { return (uint32_t)(r * 128 + (((c & 7) ^ (r & 7)) << 4)); }

// P tile: [2 atoms of 64 keys][64 rows][128 B], as the d = 128 kernel's.
CSA_DEV uint32_t swp(int r, int c, int R) {
  return (uint32_t)((c >> 3) * R * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

CSA_DEV long long shfl_i64(long long v, int src) {
  const int lo = __shfl_sync(0xffffffffu, (int)(v & 0xffffffffLL), src);
  const int hi = __shfl_sync(0xffffffffu, (int)(v >> 32), src);
  return ((long long)hi << 32) | (unsigned int)lo;
}

CSA_DEV float f32(uint32_t u) { return __uint_as_float(u); }
CSA_DEV uint32_t u32(float f) { return __float_as_uint(f); }

// Is a key with tag `tag` one of the keys of a row whose token has owner index g, visible entry
// count nv and window offsets [wlo_g, whi_g]?
CSA_DEV bool tag_valid(int32_t tag, int g, int64_t nv, int wlo_g, int whi_g) {
  if (tag < 0) return false;
  if (tag & kTagEntry) return (int64_t)(tag & kTagLow) < nv;
  if (tag & kTagWin) {
    const int o = tag & kTagLow;
    return o >= wlo_g && o <= whi_g;
  }
  return tag == g;
}

__global__ void __launch_bounds__(kThreads, 1) attend_pk_kernel(const PkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* Qs = base;                                  // [64 rows][128 B]
  uint8_t* KV = Qs + kQBytes;                          // stage s: K tile, then V tile
  uint8_t* Ps = KV + kStages * 2 * kTileBytes;         // [2 atoms][64 rows][128 B]
  int32_t* ktag = reinterpret_cast<int32_t*>(Ps + kPBytes);    // [kStages][128] key tags
  int32_t* tok_nv = ktag + kStages * kKC;              // [G] visible entries of token g
  int32_t* tok_lo = tok_nv + kMaxG;                    // [G] window offsets of token g
  int32_t* tok_hi = tok_lo + kMaxG;
  int32_t* tok_cnt = tok_hi + kMaxG;                   // [G] selected entries (sparse)
  uint64_t* bars = reinterpret_cast<uint64_t*>(tok_cnt + kMaxG);
  uint64_t* kv_full = bars;                 // [4] loaders' tags + copies of a stage (2 x 256)
  uint64_t* kv_empty = bars + kStages;      // [4] the PV reading the stage finished (commit)
  uint64_t* s_full = bars + 2 * kStages;    // [2] QK^T into S buffer finished (commit)
  uint64_t* s_free = s_full + 2;            // [2] softmax warps have read the S buffer
  uint64_t* p_full = s_free + 2;            // P written and O rescaled (8 arrivals)
  uint64_t* pv_done = p_full + 1;           // PV finished (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  float* xml = reinterpret_cast<float*>(tmem_slot + 4);  // [2 halves][64 rows][2]

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t b = blockIdx.x / p.groups;
  const int grp = blockIdx.x % p.groups;
  const int h_base = blockIdx.z * kM;
  const int i_first = grp * p.G;                         // first query of the group
  const int G_valid = min(p.G, p.Nq - i_first);          // tokens of the group that exist
  const int64_t tok0 = b * p.Nq + i_first;
  const int64_t t_first = p.q_pos0 + i_first;
  const int64_t t_last = t_first + G_valid - 1;
  const int64_t wlo = max((int64_t)0, t_first - p.W + 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 2 * kLoadThreads);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], kSoftmaxWarps);
    }
    mbar_init(p_full, kSoftmaxWarps);
    mbar_init(pv_done, 1);
    fence_mbar_init();
  }
  // The top-k counts and lists come from the kernels before this one (and a dense layer's
  // entries from the compress launch just before it).
  pdl_wait();
  // per-token parameters
  for (int g = threadIdx.x; g < p.G; g += kThreads) {
    const bool v = g < G_valid;
    const int64_t t = t_first + g;
    tok_nv[g] = v ? (int32_t)max((int64_t)0, min(p.E, (t + 1) / p.m)) : 0;
    if (v && p.W > 0) {
      tok_lo[g] = (int32_t)(max((int64_t)0, t - p.W + 1) - wlo);
      tok_hi[g] = (int32_t)(t - wlo);
    } else {
      tok_lo[g] = 1;
      tok_hi[g] = 0;
    }
    int c = 0;
    if (v && p.sparse) {
      c = p.topk_cnt[tok0 + g];
      if (c < 0 || c > p.k) {
        atomicOr(p.status, kFlagBadIndex);
        c = c < 0 ? 0 : p.k;
      }
    }
    tok_cnt[g] = c;
  }
  __syncthreads();  // barriers and per-token parameters ready: the loaders start at once
  const bool loader = warp >= kLoadWarp0 && warp < kMmaWarp;
  uint32_t tmem = 0;
  if (!loader) {
    // Q rows (token g, head h) = row g * Hp + h; zero rows for absent tokens and heads
    const int nt = warp == kMmaWarp ? kSoftmaxWarps * 32 + lane : (int)threadIdx.x;
    for (int x = nt; x < kM * 8; x += kSetupThreads) {
      const int r = x >> 3, c = x & 7;
      const int g = r / p.Hp, h = h_base + r % p.Hp;
      const bool ok = g < G_valid && h < p.H;
      cp_async_16(Qs + sw64(r, c), ok ? p.q + ((tok0 + g) * p.H + h) * kD + c * 8 : p.q,
                  ok ? 16u : 0u);
    }
    cp_async_commit();
    if (warp == kMmaWarp) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kSetupThreads) : "memory");
    tc_fence_after();
    tmem = *tmem_slot;
  }

  // the group's key list: entry slots, then the window tokens [wlo, t_last]
  const int64_t n_ent = p.sparse ? (int64_t)G_valid * p.k : (int64_t)tok_nv[G_valid - 1];
  const int64_t nwin = p.W > 0 ? t_last - wlo + 1 : 0;
  const int64_t n_keys = n_ent + nwin;
  const bool dead = (*reinterpret_cast<volatile uint32_t*>(p.status) & kFlagTimeout) != 0;
  const int nloc = dead ? 0 : (int)((n_keys + kKC - 1) / kKC);

  // softmax-warp state: lane quarter q (rows 16q .. 16q + 15), key half hf; each thread holds
  // rows r0 = 16q + g and r0 + 8
  const int gq = lane >> 2, tq = lane & 3;
  const int q = warp & 3, hf = (warp >> 2) & 1;
  const int r0 = q * 16 + gq;
  const int g0 = r0 / p.Hp, g1 = (r0 + 8) / p.Hp;  // tokens of rows r0 and r0 + 8
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  const uint32_t o_half = tmem + lane_base + kOCol + (uint32_t)(hf * kD);  // this half's O
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool sm_ok = true;

  if (loader) {
    // ------------------------------- loaders -------------------------------
    // Warp wl copies rows [16 wl, 16 wl + 16) of each chunk, four 128-byte rows per instruction
    // (8 lanes per row), after lanes 0-15 have resolved one row's source and tag each.
    const int wl = warp - kLoadWarp0;
    const int rsub = lane >> 3, cc = lane & 7;
    constexpr long long kRawBit = 1LL << 62;
    for (int it = 0; it < nloc; ++it) {
      const int s = it % kStages;
      if (it >= kStages &&
          !mbar_wait_warp(&kv_empty[s], (uint32_t)(it / kStages - 1) & 1u, p.status))
        break;
      const int i = wl * 16 + (lane & 15);
      const int64_t key = (int64_t)it * kKC + i;
      long long cd = -1;
      int32_t tag = -1;
      if (key < n_keys) {
        if (key < n_ent) {
          if (p.sparse) {
            const int g = (int)(key / p.k), jj = (int)(key - (int64_t)g * p.k);
            if (jj < tok_cnt[g]) {
              const int64_t j = p.topk_idx[(tok0 + g) * p.k + jj];
              if (j < 0 || j >= p.E) {
                atomicOr(p.status, kFlagBadIndex);  // flagged; the row is zero-filled and masked
              } else {
                cd = (b * p.E + j) * kD;
                tag = g;
              }
            }
          } else {
            cd = (b * p.E + key) * kD;
            tag = kTagEntry | (int32_t)key;
          }
        } else {
          const int64_t o = key - n_ent;
          cd = ((b * p.N + wlo + o) * kD) | kRawBit;
          tag = kTagWin | (int32_t)o;
        }
      }
      if (lane < 16) ktag[s * kKC + i] = tag;
      uint8_t* kd = KV + s * 2 * kTileBytes;
      uint8_t* vd = kd + kTileBytes;
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const int r = 4 * st + rsub;  // row within this warp's 16
        const long long c2 = shfl_i64(cd, r);
        const uint32_t off = sw64(wl * 16 + r, cc);
        const bool valid = c2 >= 0;
        const int64_t e = c2 & (kRawBit - 1);
        const bool raw = (c2 & kRawBit) != 0;
        const uint16_t* ks = valid ? (raw ? p.k_raw : p.k_cmp) + e + cc * 8 : p.k_raw;
        const uint16_t* vs = valid ? (raw ? p.v_raw : p.v_cmp) + e + cc * 8 : p.v_raw;
        cp_async_16(kd + off, ks, valid ? 16u : 0u);
        cp_async_16(vd + off, vs, valid ? 16u : 0u);
      }
      mbar_arrive(&kv_full[s]);                 // releases the tags
      cp_async_mbar_arrive_noinc(&kv_full[s]);  // arrives when the copies have landed
    }
    cp_async_wait<0>();  // never leave with copies in flight
  } else if (warp == kMmaWarp) {
    // ------------------------------- MMA issuer -------------------------------
    const uint32_t id_qk = idesc_bf16(kM, kKC, false, false);
    const uint32_t id_pv = idesc_bf16(kM, kD, false, true);
    int nq = 0, np = 0;
    long long idle0 = clock64();
    while (np < nloc) {
      bool did = false;
      if (np < nq) {
        int ready = lane == 0 ? (int)mbar_test(p_full, (uint32_t)np & 1u) : 0;
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (ready) {
          tc_fence_after();
          const int s = np % kStages;
          if (elect_one()) {
            const uint32_t pt = smem_addr(Ps);
            const uint32_t vt = smem_addr(KV + s * 2 * kTileBytes + kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kKC / 16; ++kk) {
              const uint32_t atom = kk >> 2, kin = (kk & 3) * 32;
              const uint64_t ad = smem_desc(pt + atom * kM * 128 + kin, 16, 1024, kSwizzle128B);
              // V rows are keys (the K dimension) with d contiguous: MN-major B of one 64-column
              // atom, 8-key groups 1024 bytes apart
              const uint64_t bd = smem_desc(vt + kk * 16 * 128, kKC * 128, 1024, kSwizzle128B);
              umma_bf16(tmem + kOCol + atom * kD, ad, bd, id_pv,
                        (np > 0 || (kk & 3) > 0) ? 1u : 0u);
            }
            umma_commit(&kv_empty[s]);
            umma_commit(pv_done);
          }
          __syncwarp();
          ++np;
          did = true;
        }
      }
      if (nq < nloc) {
        const int s = nq % kStages, sb = nq & 1;
        int ready = 0;
        if (lane == 0)
          ready = mbar_test(&kv_full[s], (uint32_t)(nq / kStages) & 1u) &&
                  (nq < 2 || mbar_test(&s_free[sb], (uint32_t)((nq >> 1) - 1) & 1u));
        ready = __shfl_sync(0xffffffffu, ready, 0);
        if (ready) {
          fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
          tc_fence_after();
          if (elect_one()) {
            const uint32_t kt = smem_addr(KV + s * 2 * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint32_t kin = kk * 32;
              const uint64_t ad = smem_desc(smem_addr(Qs) + kin, 16, 1024, kSwizzle128B);
              const uint64_t bd = smem_desc(kt + kin, 16, 1024, kSwizzle128B);
              umma_bf16(tmem + (uint32_t)(sb * kKC), ad, bd, id_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[sb]);
          }
          __syncwarp();
          ++nq;
          did = true;
        }
      }
      if (did) {
        idle0 = clock64();
      } else if (clock64() - idle0 > kWaitBudgetCycles) {
        if (lane == 0) atomicOr(p.status, kFlagTimeout);
        break;
      }
    }
  } else {
    // ------------------------------- softmax -------------------------------
    // Keys [64 hf, 64 hf + 64) of every chunk with their own running maximum and sum; the two
    // key halves accumulate into separate O accumulators that are combined at the end. Rows r0
    // and r0 + 8 belong to tokens g0 and g1; a key counts for a row when its tag is that row's.
    const int64_t nv0 = tok_nv[g0], nv1 = tok_nv[g1];
    const int lo0 = tok_lo[g0], hi0 = tok_hi[g0], lo1 = tok_lo[g1], hi1 = tok_hi[g1];
    for (int it = 0; it < nloc; ++it) {
      const int sb = it & 1, s = it % kStages;
      if (!mbar_wait_warp(&s_full[sb], (uint32_t)(it >> 1) & 1u, p.status)) {
        sm_ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[32];  // r[4i + e]: row r0, key 8i + 2tq + e of the half; r[4i + 2 + e]: row r0 + 8
      tmem_ld_16x256b_x8(tmem + lane_base + (uint32_t)(sb * kKC + hf * kHalf), r);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);
      // the stage's tags (the phase completed before S did; acquire the loaders' stores)
      if (!mbar_wait_warp(&kv_full[s], (uint32_t)(it / kStages) & 1u, p.status)) {
        sm_ok = false;
        break;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int2 tg = *reinterpret_cast<const int2*>(&ktag[s * kKC + hf * kHalf + 8 * i + 2 * tq]);
        const int32_t tgs[2] = {tg.x, tg.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (!tag_valid(tgs[e], g0, nv0, lo0, hi0)) r[4 * i + e] = u32(-INFINITY);
          if (!tag_valid(tgs[e], g1, nv1, lo1, hi1)) r[4 * i + 2 + e] = u32(-INFINITY);
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        mx0 = fmaxf(mx0, fmaxf(f32(r[4 * i]), f32(r[4 * i + 1])));
        mx1 = fmaxf(mx1, fmaxf(f32(r[4 * i + 2]), f32(r[4 * i + 3])));
      }
#pragma unroll
      for (int x = 1; x < 4; x <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
      }
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // true also when the old reference is -inf and the new one finite; false if both are -inf
      const bool need0 = (mn0 - m0) * kLog2e > kRescaleLog2;
      const bool need1 = (mn1 - m1) * kLog2e > kRescaleLog2;
      const bool rescale = __any_sync(0xffffffffu, need0 || need1);
      float c0 = 1.f, c1 = 1.f;
      if (rescale) {
        c0 = need0 ? exp2f((m0 - mn0) * kLog2e) : 1.f;
        c1 = need1 ? exp2f((m1 - mn1) * kLog2e) : 1.f;
        l0 *= c0;
        l1 *= c1;
        if (need0) m0 = mn0;
        if (need1) m1 = mn1;
      }
      const float nb0 = m0 == -INFINITY ? 0.f : -m0 * kLog2e;
      const float nb1 = m1 == -INFINITY ? 0.f : -m1 * kLog2e;
      uint32_t pk[16];
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float p00 = ex2_approx(fmaf(f32(r[4 * i + 0]), kLog2e, nb0));
        const float p01 = ex2_approx(fmaf(f32(r[4 * i + 1]), kLog2e, nb0));
        const float p10 = ex2_approx(fmaf(f32(r[4 * i + 2]), kLog2e, nb1));
        const float p11 = ex2_approx(fmaf(f32(r[4 * i + 3]), kLog2e, nb1));
        rs0 += p00 + p01;
        rs1 += p10 + p11;
        pk[2 * i] = pack_bf16x2(p00, p01);
        pk[2 * i + 1] = pack_bf16x2(p10, p11);
      }
      l0 += rs0;
      l1 += rs1;
      if (it > 0) {
        // PV(it - 1) finished: P may be rewritten and O holds every PV so far
        if (!mbar_wait_warp(pv_done, (uint32_t)(it - 1) & 1u, p.status)) {
          sm_ok = false;
          break;
        }
        tc_fence_after();
        if (rescale) {
#pragma unroll
          for (int part = 0; part < kD / 32; ++part) {
            uint32_t ov[16];
            const uint32_t oa = o_half + (uint32_t)(part * 32);
            tmem_ld_16x256b_x4(oa, ov);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              ov[4 * i + 0] = u32(f32(ov[4 * i + 0]) * c0);
              ov[4 * i + 1] = u32(f32(ov[4 * i + 1]) * c0);
              ov[4 * i + 2] = u32(f32(ov[4 * i + 2]) * c1);
              ov[4 * i + 3] = u32(f32(ov[4 * i + 3]) * c1);
            }
            tmem_st_16x256b_x4(oa, ov);
          }
          tmem_st_wait();
        }
      }
      // P rows 16q .. 16q + 15, keys 64 hf .. 64 hf + 63 (atom hf, 16-byte chunks 0-7): each
      // stmatrix.x4 stores two chunks x two 8-row halves; lane l addresses row l % 8 (+ 8 for
      // the odd matrices) of chunk 2c + l / 16.
      {
        const int mrow = q * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int mchunk = lane >> 4;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          stmatrix_x4(smem_addr(Ps + swp(mrow, 8 * hf + 2 * c + mchunk, kM)), pk[4 * c],
                      pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      }
      fence_proxy_async_smem();  // P (generic stores) -> tensor-core reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (sm_ok && nloc > 0)
      sm_ok = mbar_wait_warp(pv_done, (uint32_t)(nloc - 1) & 1u, p.status);
#pragma unroll
    for (int x = 1; x < 4; x <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, x);
      l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }
    if (tq == 0) {  // this half's (max, sum) of both rows, for the other half
      xml[(hf * kM + r0) * 2 + 0] = m0;
      xml[(hf * kM + r0) * 2 + 1] = l0;
      xml[(hf * kM + r0 + 8) * 2 + 0] = m1;
      xml[(hf * kM + r0 + 8) * 2 + 1] = l1;
    }
  }

  __syncthreads();
  // Combine the two key halves: warp (q, hf) produces output columns [32 hf, 32 hf + 32) of rows
  // r0 and r0 + 8 from both O accumulators, weighted to the common maximum.
  const bool smx = warp < kSoftmaxWarps;
  uint32_t o[16];
  float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
  if (smx) {
    const float ma0 = xml[(0 * kM + r0) * 2], la0 = xml[(0 * kM + r0) * 2 + 1];
    const float mb0 = xml[(1 * kM + r0) * 2], lb0 = xml[(1 * kM + r0) * 2 + 1];
    const float ma1 = xml[(0 * kM + r0 + 8) * 2], la1 = xml[(0 * kM + r0 + 8) * 2 + 1];
    const float mb1 = xml[(1 * kM + r0 + 8) * 2], lb1 = xml[(1 * kM + r0 + 8) * 2 + 1];
    M0 = fmaxf(ma0, mb0);
    M1 = fmaxf(ma1, mb1);
    const float wa0 = ma0 == -INFINITY ? 0.f : exp2f((ma0 - M0) * kLog2e);
    const float wb0 = mb0 == -INFINITY ? 0.f : exp2f((mb0 - M0) * kLog2e);
    const float wa1 = ma1 == -INFINITY ? 0.f : exp2f((ma1 - M1) * kLog2e);
    const float wb1 = mb1 == -INFINITY ? 0.f : exp2f((mb1 - M1) * kLog2e);
    L0 = wa0 * la0 + wb0 * lb0;
    L1 = wa1 * la1 + wb1 * lb1;
#pragma unroll
    for (int x = 0; x < 16; ++x) o[x] = 0u;
    if (sm_ok && nloc > 0) {
      tc_fence_after();
      uint32_t oa[16], ob[16];
      const uint32_t col = tmem + lane_base + kOCol + (uint32_t)(hf * 32);
      tmem_ld_16x256b_x4(col, oa);       // key half 0, output columns 32 hf ..
      tmem_ld_16x256b_x4(col + kD, ob);  // key half 1
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        o[4 * i + 0] = u32(wa0 * f32(oa[4 * i + 0]) + wb0 * f32(ob[4 * i + 0]));
        o[4 * i + 1] = u32(wa0 * f32(oa[4 * i + 1]) + wb0 * f32(ob[4 * i + 1]));
        o[4 * i + 2] = u32(wa1 * f32(oa[4 * i + 2]) + wb1 * f32(ob[4 * i + 2]));
        o[4 * i + 3] = u32(wa1 * f32(oa[4 * i + 3]) + wb1 * f32(ob[4 * i + 3]));
      }
    }
  }
  // Every role is done with tensor memory and the pipeline buffers.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (smx) {
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    const int ha = h_base + r0 % p.Hp, hb = h_base + (r0 + 8) % p.Hp;
    const bool va = g0 < G_valid && ha < p.H, vb = g1 < G_valid && hb < p.H;
    const int64_t ra = (tok0 + g0) * p.H + ha, rb = (tok0 + g1) * p.H + hb;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d0 = hf * 32 + 8 * i + 2 * tq;
      if (va)
        *reinterpret_cast<uint32_t*>(p.out + ra * kD + d0) =
            pack_bf16x2(f32(o[4 * i]) * inv0, f32(o[4 * i + 1]) * inv0);
      if (vb)
        *reinterpret_cast<uint32_t*>(p.out + rb * kD + d0) =
            pack_bf16x2(f32(o[4 * i + 2]) * inv1, f32(o[4 * i + 3]) * inv1);
    }
    if (p.lse != nullptr && tq == 0 && hf == 0) {
      if (va) p.lse[ra] = L0 > 0.f ? M0 + logf(L0) : -INFINITY;
      if (vb) p.lse[rb] = L1 > 0.f ? M1 + logf(L1) : -INFINITY;
    }
  }
}

}  // namespace

// Packed prefill launch for d = 64: G = 64 / Hp query tokens of one sequence per CTA.
cudaError_t launch_attend_pk(const AttendArgs& a, uint32_t* status, cudaStream_t stream) {
  if (a.d != kD || a.paged) return cudaErrorInvalidValue;
  PkParams prm;
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
  int hp = 1;
  while (hp < a.H && hp < kM) hp <<= 1;
  prm.Hp = hp;
  prm.G = kM / hp;
  prm.groups = (a.Nq + prm.G - 1) / prm.G;
  prm.sparse = a.topk_idx != nullptr;
  prm.status = status;
  if (prm.sparse && (a.k < 1 || (int64_t)prm.G * a.k > (int64_t)kTagWin)) return cudaErrorInvalidValue;
  if (!prm.sparse && a.E >= (int64_t)kTagWin) return cudaErrorInvalidValue;
  auto kern = attend_pk_kernel;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int hgroups = (a.H + kM - 1) / kM;
  ProfScope prof(stream, prm.sparse ? "csa_attend" : "hca_attend");
  return launch_ex(kern, dim3((unsigned)(a.B * prm.groups), 1u, (unsigned)hgroups),
                   dim3(kThreads), kSmemBytes, stream, 1u, prm);
}

}  // namespace csa
