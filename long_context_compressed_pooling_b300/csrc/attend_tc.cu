// CSA sparse attention and HCA dense attention on the 5th-generation tensor cores (tcgen05), for
// head dim 128.
//
// Lighthouse "deep deepseek v4 release" 八.3: CSA attends to the top-k selected compressed
// entries plus a sliding-window branch of n_win raw tokens; HCA attends densely to every
// compressed entry plus the same window. One softmax spans a query's entries and window tokens;
// logits are q.k (the 1/sqrt(d) is folded into q).
//
// MQA: the H query heads of a token share one K/V head, so one CTA owns one query token and 64
// heads, which form the M = 64 side of both contractions:
//   S[64 heads, 128 keys]  = Q[64, 128 d] . K_chunk^T        (A = Q, B = K rows; both K-major)
//   O[64 heads, 128 d]    += P[64, 128 keys] . V_chunk        (A = P, B = V rows read MN-major)
// S and O live in tensor memory (S double-buffered: 2 x 128 columns; two O accumulators of 128
// columns, one per key half). With M = 64 the accumulator rows 16q..16q+15 sit in lanes
// 32q..32q+15, so a softmax warp reads its 16 rows with the 16x256b load, which hands every
// thread two rows in the m16n8 fragment layout.
//
// Warp roles (576 threads, one CTA per SM):
//   warps 0-7  softmax: warp w reads rows 16(w % 4) .. +15 of key half w / 4 of S, masks, runs an
//              online softmax with its own running maximum per key half, writes P (bf16) to
//              shared memory, and rescales its O accumulator in tensor memory only when the
//              running maximum has risen by more than 2^8 (the reference maximum of a row only
//              moves then, so P stays below 2^8 and the normalisation at the end uses the same
//              reference); at the end the two key halves are combined, normalised and stored;
//   warps 8-15 loaders: gather the key rows of each 128-key chunk (selected entries or window
//              tokens; through the block table and the ring for a paged cache) with 16-byte
//              cp.async into 128-byte-swizzled K and V tiles, two 256-byte rows per warp
//              instruction, and write a validity bit per key (missing keys, out-of-range indices
//              and unmapped pages are zero-filled and masked); each loader thread arrives on the
//              stage's barrier twice: at once (releasing the mask bits) and when its copies land
//              (cp.async.mbarrier.arrive);
//   warp 16    tensor-memory allocation and the QK^T MMAs of each chunk once its K/V rows have
//              landed and an S buffer is free (one elected lane of the converged warp);
//   warp 17    the PV MMAs of each chunk once its P is written: a tcgen05.mma takes ~100 cycles
//              to issue from one thread, so the two contractions have an issuing warp each.
// Three K/V stages (64 KB each) and one P buffer; every mbarrier wait is bounded.
//
// Prefill (one split per token) runs persistent CTAs, one per SM, each walking the (token, head
// group) items blockIdx.y, blockIdx.y + gridDim.y, ...: the loaders run on into the next item's
// chunks while the softmax warps finish the current one, so a token's start no longer waits for
// the previous token's tail (prefill attention 1.60 -> 1.47 ms on csa_prefill_8k_of_128k).
//
// Decode splits a token's key chunks over several CTAs: the splits of a token form a cluster and
// merge their (max, sum, unnormalised O) through distributed shared memory, or (more than 16
// splits) through the workspace and a separate merge kernel, as in the mma.sync kernel.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kD = 128;            // head dim
constexpr int kM = 64;             // heads per CTA (MMA M)
constexpr int kKC = 128;           // keys per chunk (N of QK^T, K of PV)
constexpr int kHalf = kKC / 2;     // keys per softmax warp (and per O accumulator)
constexpr int kStages = 3;         // K/V stages
constexpr int kSoftmaxWarps = 8;   // warps 0-7: lane quarter w % 4, key half w / 4
constexpr int kLoadWarp0 = 8;      // warps 8-15
constexpr int kLoadWarps = 8;
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kMmaWarp = 16;      // QK^T issuer, tensor-memory allocation
constexpr int kPvWarp = 17;       // PV issuer
constexpr int kThreads = 576;
constexpr int kSetupThreads = 32 * (kSoftmaxWarps + 2);  // softmax warps + both MMA warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;    // O accumulators: key half 0 at [256, 384), half 1 at [384, 512)
constexpr int kQBytes = kM * kD * 2;        // 16 KB
constexpr int kTileBytes = kKC * kD * 2;    // 32 KB (one K or V tile)
constexpr int kPBytes = kM * kKC * 2;       // 16 KB
constexpr int kMaxClusterSplits = 16;
constexpr int kPStride = kD + 4;            // padded row of a parked partial output (floats)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kNumBars = 16;
constexpr size_t kSmemBytes = 1024 + kQBytes + (size_t)kStages * 2 * kTileBytes + kPBytes +
                              kNumBars * 8 + 16 + kStages * 4 * 4 + 2 * kM * 2 * 4;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct TcParams {
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
  float* ws_ml;  // [n_splits, tokens, H, 2] reference maximum and sum
  int64_t E, N, q_pos0;
  int64_t fresh_from;  // dense: entries below it may be read before the predecessor completes
  // paged cache (block_table != null): entry j of sequence b is row (page << page_shift) +
  // (j & page_mask) of the entry pools, page = block_table[b][j >> page_shift]; window token at
  // position pos is row b * kRingTokens + (pos & (kRingTokens - 1)) of the raw rings
  const int32_t* block_table;
  int max_blocks, n_pages, page_shift;
  int k, m, W, Nq, H, n_splits, tokens;
  int sparse;
  int cluster_merge;
  uint32_t* status;
};

// Byte offset of 16-byte chunk c (0..15) of row r in a 128-byte-swizzled K-major tile of R rows
// and 128 bf16 columns: two 64-column atoms of R x 128 B, chunk index XOR (row mod 8).
CSA_DEV uint32_t sw128(int r, int c, int R) {
  return (uint32_t)((c >> 3) * R * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

CSA_DEV long long shfl_i64(long long v, int src) {
  const int lo = __shfl_sync(0xffffffffu, (int)(v & 0xffffffffLL), src);
  const int hi = __shfl_sync(0xffffffffu, (int)(v >> 32), src);
  return ((long long)hi << 32) | (unsigned int)lo;
}

CSA_DEV float f32(uint32_t u) { return __uint_as_float(u); }
CSA_DEV uint32_t u32(float f) { return __float_as_uint(f); }

// One work item: query token `tok` and heads [h_base, h_base + 64), and this CTA's chunks of
// its key list.
struct Item {
  int64_t tok, b, t, n_sel, w0, n_keys;
  int h_base, c_begin, nloc;
};

// kPersist: one CTA per SM walks the items blockIdx.y, blockIdx.y + gridDim.y, ... (no split of
// a token's keys). Every role runs its own loop over the same items and the pipeline's counters
// (stage, S buffer, barrier phases) run on across them, so the loaders fetch the next item's
// first chunks while the softmax warps finish this one; the QK^T warp reloads Q once the last
// QK^T of the previous item has finished, and the first PV of an item waits until the softmax
// warps have read the previous item's O. Otherwise the CTA owns one item (and one split of it).
template <bool kPersist>
__global__ void __launch_bounds__(kThreads, 1) attend_tc_kernel(const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* Qs = base;                                  // [2 atoms][64 rows][128 B]
  uint8_t* KV = Qs + kQBytes;                          // stage s: K tile, then V tile
  uint8_t* Ps = KV + kStages * 2 * kTileBytes;         // [2 atoms][64 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(Ps + kPBytes);
  uint64_t* kv_full = bars;        // [3] loaders' mask words + copies of a stage (2 x 128)
  uint64_t* kv_empty = bars + 3;   // [3] the PV reading the stage finished (commit)
  uint64_t* s_full = bars + 6;     // [2] QK^T into S buffer finished (commit)
  uint64_t* s_free = bars + 8;     // [2] softmax warps have read the S buffer (8 arrivals)
  uint64_t* p_full = bars + 10;    // P written and O rescaled (8 arrivals)
  uint64_t* pv_done = bars + 11;   // PV finished (commit); P may be rewritten, O read
  uint64_t* o_free = bars + 12;    // persistent: the softmax warps have read O (8 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  uint32_t* sm_abort = tmem_slot + 1;                  // persistent: a softmax wait failed
  uint32_t* kmask = tmem_slot + 4;                     // [3][4] validity bits of the 128 keys
  float* xml = reinterpret_cast<float*>(kmask + kStages * 4);  // [2 halves][64 rows][2]

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = p.cluster_merge ? (int)cluster_ctarank() : (int)blockIdx.x;
  // item i: token i / groups, heads (i % groups) * 64 ..
  const int groups = (p.H + kM - 1) / kM;
  const int64_t n_items = (int64_t)p.tokens * groups;
  const int64_t item0 = kPersist ? (int64_t)blockIdx.y : (int64_t)blockIdx.y * groups + blockIdx.z;
  // a non-persistent CTA's loops run once, over item0, as the compiler can see
  const int64_t item_step = kPersist ? (int64_t)gridDim.y : 1;
  const int64_t item_end = kPersist ? n_items : item0 + 1;

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
    mbar_init(o_free, kSoftmaxWarps);
    *sm_abort = 0u;
    fence_mbar_init();
  }
  __syncthreads();  // barriers initialised: the loaders start their copies at once
  const bool loader = warp >= kLoadWarp0 && warp < kMmaWarp;
  uint32_t tmem = 0;
  if (!loader) {
    // Q tile of the first item's heads (zero rows past H; Q is an input of this call) and the
    // tensor memory, by the softmax and MMA warps while the loaders' first copies fly
    const int64_t tok0 = kPersist ? item0 / groups : (int64_t)blockIdx.y;
    const int hb0 = kPersist ? (int)(item0 % groups) * kM : (int)blockIdx.z * kM;
    const int nt = warp >= kMmaWarp ? (kSoftmaxWarps + warp - kMmaWarp) * 32 + lane
                                    : (int)threadIdx.x;
    for (int x = nt; x < kM * 16; x += kSetupThreads) {
      const int r = x >> 4, c = x & 15;
      const bool ok = hb0 + r < p.H;
      cp_async_16(Qs + sw128(r, c, kM), ok ? p.q + (tok0 * p.H + hb0 + r) * kD + c * 8 : p.q,
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
  // Top-k lists come from the preceding kernels; a dense launch defers the wait until its
  // loaders reach an entry at or above fresh_from (raw window rows and Q are inputs).
  const bool early = !p.sparse && p.fresh_from > 0;
  if (!early) pdl_wait();

  // After a wait has timed out anywhere on the device, later CTAs skip their work instead of
  // timing out one after another.
  const bool dead = (*reinterpret_cast<volatile uint32_t*>(p.status) & kFlagTimeout) != 0;
  auto item_at = [&](int64_t i) {
    Item I;
    if constexpr (kPersist) {
      I.tok = i / groups;
      I.h_base = (int)(i % groups) * kM;
    } else {  // the CTA's one item (64-bit division is emulated: none here)
      I.tok = blockIdx.y;
      I.h_base = (int)blockIdx.z * kM;
    }
    I.b = I.tok / p.Nq;
    I.t = p.q_pos0 + I.tok % p.Nq;
    if (p.sparse) {
      int64_t n = p.topk_cnt[I.tok];
      if (n < 0 || n > p.k) {
        if (threadIdx.x == 0) atomicOr(p.status, kFlagBadIndex);
        n = n < 0 ? 0 : p.k;
      }
      I.n_sel = n;
    } else {
      I.n_sel = max((int64_t)0, min(p.E, (I.t + 1) / p.m));
    }
    I.w0 = max((int64_t)0, I.t - p.W + 1);
    I.n_keys = I.n_sel + (p.W > 0 ? (I.t - I.w0 + 1) : 0);
    const int n_chunks = (int)((I.n_keys + kKC - 1) / kKC);
    I.c_begin = n_chunks * split / p.n_splits;
    I.nloc = dead ? 0 : n_chunks * (split + 1) / p.n_splits - I.c_begin;
    return I;
  };

  // softmax-warp state: lane quarter q (rows 16q .. 16q + 15), key half hf; each thread holds
  // rows r0 = 16q + g and r0 + 8
  const int g = lane >> 2, tq = lane & 3;
  const int q = warp & 3, hf = (warp >> 2) & 1;
  const int r0 = q * 16 + g;
  const uint32_t lane_base = (uint32_t)(q * 32) << 16;
  const uint32_t o_half = tmem + lane_base + kOCol + (uint32_t)(hf * kD);  // this half's O
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool sm_ok = true;
  int sm_nloc = 0;  // a softmax warp's chunks of its (last) item
  const int dc = hf * 64;  // a softmax warp's output columns

  // The two key halves of an item combined (softmax warps, after both halves' (max, sum) are in
  // xml): warp (q, hf) produces output columns [64 hf, 64 hf + 64) of rows r0 and r0 + 8 from
  // both O accumulators, weighted to the common maximum.
  auto combine = [&](bool read_o, uint32_t(&o)[32], float& M0, float& M1, float& L0, float& L1) {
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
    for (int x = 0; x < 32; ++x) o[x] = 0u;
    if (read_o) {
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t oa[16], ob[16];
        const uint32_t col = tmem + lane_base + kOCol + (uint32_t)(hf * 64 + part * 32);
        tmem_ld_16x256b_x4(col, oa);       // key half 0, output columns 64 hf + 32 part ..
        tmem_ld_16x256b_x4(col + kD, ob);  // key half 1
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int x = 16 * part + 4 * i;
          o[x + 0] = u32(wa0 * f32(oa[4 * i + 0]) + wb0 * f32(ob[4 * i + 0]));
          o[x + 1] = u32(wa0 * f32(oa[4 * i + 1]) + wb0 * f32(ob[4 * i + 1]));
          o[x + 2] = u32(wa1 * f32(oa[4 * i + 2]) + wb1 * f32(ob[4 * i + 2]));
          o[x + 3] = u32(wa1 * f32(oa[4 * i + 3]) + wb1 * f32(ob[4 * i + 3]));
        }
      }
    }
  };
  // normalised bf16 output (and log-sum-exp) of rows r0, r0 + 8 of a whole (unsplit) item
  auto store_out = [&](int64_t tok, int h_base, const uint32_t(&o)[32], float M0, float M1,
                       float L0, float L1) {
    const int h0 = h_base + r0, h1 = h0 + 8;
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d0 = dc + 8 * i + 2 * tq;
      if (h0 < p.H)
        *reinterpret_cast<uint32_t*>(p.out + (tok * p.H + h0) * kD + d0) =
            pack_bf16x2(f32(o[4 * i]) * inv0, f32(o[4 * i + 1]) * inv0);
      if (h1 < p.H)
        *reinterpret_cast<uint32_t*>(p.out + (tok * p.H + h1) * kD + d0) =
            pack_bf16x2(f32(o[4 * i + 2]) * inv1, f32(o[4 * i + 3]) * inv1);
    }
    if (p.lse != nullptr && tq == 0 && hf == 0) {
      if (h0 < p.H) p.lse[tok * p.H + h0] = L0 > 0.f ? M0 + logf(L0) : -INFINITY;
      if (h1 < p.H) p.lse[tok * p.H + h1] = L1 > 0.f ? M1 + logf(L1) : -INFINITY;
    }
  };

  if (loader) {
    // ------------------------------- loaders -------------------------------
    // Warp wl copies rows [16 wl, 16 wl + 16) of each chunk, two rows per instruction: lanes
    // 0-15 and 16-31 each copy the 16 chunks of one 256-byte row (coalesced).
    const int wl = warp - kLoadWarp0;
    const int h = lane >> 4, cc = lane & 15;
    constexpr long long kRawBit = 1LL << 62;
    bool waited = !early;
    bool run = true;
    int gc = 0;  // this CTA's chunks so far, over all its items
    for (int64_t ii = item0; ii < item_end && run; ii += item_step) {
      const Item I = item_at(ii);
      for (int it = 0; it < I.nloc; ++it, ++gc) {
        const int s = gc % kStages;
        const int64_t k0 = (int64_t)(I.c_begin + it) * kKC;
        if (!waited && k0 < I.n_sel && k0 + kKC > p.fresh_from) {
          pdl_wait();
          waited = true;
        }
        if (gc >= kStages &&
            !mbar_wait_warp(&kv_empty[s], (uint32_t)(gc / kStages - 1) & 1u, p.status)) {
          run = false;
          break;
        }
        // source row of row 16 wl + lane % 16 (element offset; bit 62 = raw window token, -1 =
        // none); lanes 16-31 repeat lanes 0-15
        const int i = wl * 16 + (lane & 15);
        const int64_t key = k0 + i;
        long long cd = -1;
        if (key < I.n_keys) {
          if (key < I.n_sel) {
            const int64_t j = p.sparse ? (int64_t)p.topk_idx[I.tok * p.k + key] : key;
            if (j < 0 || j >= p.E) {
              atomicOr(p.status, kFlagBadIndex);  // flagged; the row is zero-filled and masked
            } else if (p.block_table) {
              const int64_t blk = j >> p.page_shift;
              const int pg = blk < p.max_blocks ? p.block_table[I.b * p.max_blocks + blk] : -1;
              if (pg < 0 || pg >= p.n_pages)
                atomicOr(p.status, kFlagBadIndex);  // unmapped page: zero-filled and masked
              else
                cd = (((int64_t)pg << p.page_shift) + (j & ((1 << p.page_shift) - 1))) * kD;
            } else {
              cd = (I.b * p.E + j) * kD;
            }
          } else {
            const int64_t pos = I.w0 + (key - I.n_sel);
            cd = ((p.block_table ? I.b * kRingTokens + (pos & (kRingTokens - 1))
                                 : I.b * p.N + pos) *
                  kD) |
                 kRawBit;
          }
        }
        const uint32_t vbits = __ballot_sync(0xffffffffu, cd >= 0);
        if (lane == 0)
          reinterpret_cast<uint16_t*>(kmask)[s * 8 + wl] = (uint16_t)(vbits & 0xFFFFu);
        uint8_t* kd = KV + s * 2 * kTileBytes;
        uint8_t* vd = kd + kTileBytes;
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const int r = 2 * st + h;  // row within this warp's 16
          const long long c2 = shfl_i64(cd, r);
          const uint32_t off = sw128(wl * 16 + r, cc, kKC);
          const bool valid = c2 >= 0;
          const int64_t e = c2 & (kRawBit - 1);
          const bool raw = (c2 & kRawBit) != 0;
          const uint16_t* ks = valid ? (raw ? p.k_raw : p.k_cmp) + e + cc * 8 : p.k_raw;
          const uint16_t* vs = valid ? (raw ? p.v_raw : p.v_cmp) + e + cc * 8 : p.v_raw;
          cp_async_16(kd + off, ks, valid ? 16u : 0u);
          cp_async_16(vd + off, vs, valid ? 16u : 0u);
        }
        mbar_arrive(&kv_full[s]);                 // releases the mask word
        cp_async_mbar_arrive_noinc(&kv_full[s]);  // arrives when the copies have landed
      }
    }
    cp_async_wait<0>();  // never leave with copies in flight
  } else if (warp == kMmaWarp) {
    // ------------------------------- QK^T issuer -------------------------------
    // One tcgen05.mma takes ~100 cycles to issue from one thread, so QK^T and PV have a warp
    // each: QK^T of the next chunk never waits behind the PV of the current one.
    const uint32_t id_qk = idesc_bf16(kM, kKC, false, false);
    bool run = true;
    int gc = 0;
    int64_t q_item = item0;  // the item whose Q tile is in shared memory
    for (int64_t ii = item0; ii < item_end && run; ii += item_step) {
      const Item I = item_at(ii);
      if constexpr (kPersist) {
        const int64_t nx = ii + item_step;
        if (lane == 0 && nx < n_items) {  // the next item's Q on its way into L2
          const int nh = (int)(nx % groups) * kM;
          prefetch_l2(p.q + ((nx / groups) * p.H + nh) * kD, (uint32_t)(min(kM, p.H - nh) * kD * 2));
        }
        if (I.nloc > 0 && q_item != ii) {
          // the previous chunk's QK^T has finished reading Q: this item's Q replaces it
          if (gc > 0 &&
              !mbar_wait_warp(&s_full[(gc - 1) & 1], (uint32_t)((gc - 1) >> 1) & 1u, p.status))
            break;
          for (int x = lane; x < kM * 16; x += 32) {
            const int r = x >> 4, c = x & 15;
            const bool ok = I.h_base + r < p.H;
            cp_async_16(Qs + sw128(r, c, kM),
                        ok ? p.q + (I.tok * p.H + I.h_base + r) * kD + c * 8 : p.q,
                        ok ? 16u : 0u);
          }
          cp_async_commit();
          cp_async_wait<0>();
          fence_proxy_async_smem();  // Q (cp.async writes) -> tensor-core reads
          __syncwarp();
          q_item = ii;
        }
      }
      for (int nq = 0; nq < I.nloc; ++nq, ++gc) {
        const int s = gc % kStages, sb = gc & 1;
        if (!mbar_wait_warp(&kv_full[s], (uint32_t)(gc / kStages) & 1u, p.status) ||
            (gc >= 2 && !mbar_wait_warp(&s_free[sb], (uint32_t)((gc >> 1) - 1) & 1u, p.status))) {
          run = false;
          break;
        }
        fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
        tc_fence_after();
        // descriptors of the first K step, built by the whole (converged) warp; a step's
        // descriptor adds its byte offset / 16 to the start-address field
        const uint64_t qd = smem_desc(smem_addr(Qs), 16, 1024, kSwizzle128B);
        const uint64_t kd = smem_desc(smem_addr(KV + s * 2 * kTileBytes), 16, 1024, kSwizzle128B);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t atom = kk >> 2, kin = (kk & 3) * 32;
            umma_bf16(tmem + (uint32_t)(sb * kKC), qd + ((atom * kM * 128 + kin) >> 4),
                      kd + ((atom * kKC * 128 + kin) >> 4), id_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[sb]);
        }
        __syncwarp();
      }
    }
  } else if (warp == kPvWarp) {
    // ------------------------------- PV issuer -------------------------------
    const uint32_t id_pv = idesc_bf16(kM, kD, false, true);
    bool run = true;
    int gc = 0, nprev = 0;  // chunks so far; items with chunks so far
    for (int64_t ii = item0; ii < item_end && run; ii += item_step) {
      const Item I = item_at(ii);
      // the first PV of an item overwrites O: the softmax warps have read the previous one's
      if (kPersist && I.nloc > 0 && nprev > 0 &&
          !mbar_wait_warp(o_free, (uint32_t)(nprev - 1) & 1u, p.status))
        break;
      for (int np = 0; np < I.nloc; ++np, ++gc) {
        const int s = gc % kStages;
        // P of the chunk is written (and its stage's V rows landed before its S existed)
        if (!mbar_wait_warp(p_full, (uint32_t)gc & 1u, p.status) ||
            !mbar_wait_warp(&kv_full[s], (uint32_t)(gc / kStages) & 1u, p.status)) {
          run = false;
          break;
        }
        fence_proxy_async_smem();
        tc_fence_after();
        const uint64_t pd = smem_desc(smem_addr(Ps), 16, 1024, kSwizzle128B);
        // V rows are keys (the K dimension) with d contiguous: MN-major B, 64-column atoms
        // kKC * 128 bytes apart, 8-key groups 1024 bytes apart.
        const uint64_t vd = smem_desc(smem_addr(KV + s * 2 * kTileBytes + kTileBytes), kKC * 128,
                                      1024, kSwizzle128B);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kKC / 16; ++kk) {
            const uint32_t atom = kk >> 2, kin = (kk & 3) * 32;
            // keys 0-63 accumulate into O half 0, keys 64-127 into O half 1
            umma_bf16(tmem + kOCol + atom * kD, pd + ((atom * kM * 128 + kin) >> 4),
                      vd + ((kk * 16 * 128) >> 4), id_pv, (np > 0 || (kk & 3) > 0) ? 1u : 0u);
          }
          umma_commit(&kv_empty[s]);
          umma_commit(pv_done);
        }
        __syncwarp();
      }
      if (I.nloc > 0) ++nprev;
    }
  } else {
    // ------------------------------- softmax -------------------------------
    // Keys [64 hf, 64 hf + 64) of every chunk, with their own running maximum and sum; the two
    // key halves accumulate into separate O accumulators that are combined at the end.
    int gc = 0;
    for (int64_t ii = item0; ii < item_end; ii += item_step) {
      const Item I = item_at(ii);
      sm_nloc = I.nloc;
      m0 = -INFINITY;
      m1 = -INFINITY;
      l0 = 0.f;
      l1 = 0.f;
      for (int it = 0; it < I.nloc; ++it, ++gc) {
        const int sb = gc & 1, s = gc % kStages;
        if (!mbar_wait_warp(&s_full[sb], (uint32_t)(gc >> 1) & 1u, p.status)) {
          sm_ok = false;
          break;
        }
        tc_fence_after();
        uint32_t r[32];  // r[4i + e]: row r0, key 8i + 2tq + e of the half; r[4i + 2 + e]: r0 + 8
        tmem_ld_16x256b_x8(tmem + lane_base + (uint32_t)(sb * kKC + hf * kHalf), r);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);
        // the stage's mask words (the phase completed before S did; acquire the loaders' stores)
        if (!mbar_wait_warp(&kv_full[s], (uint32_t)(gc / kStages) & 1u, p.status)) {
          sm_ok = false;
          break;
        }
        const uint32_t mlo = kmask[s * 4 + 2 * hf], mhi = kmask[s * 4 + 2 * hf + 1];
        if ((mlo & mhi) != 0xffffffffu) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const uint32_t bit = (((i < 4) ? mlo : mhi) >> ((8 * i + 2 * tq + e) & 31)) & 1u;
              if (!bit) {
                r[4 * i + e] = u32(-INFINITY);
                r[4 * i + 2 + e] = u32(-INFINITY);
              }
            }
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
        // true also when the old reference is -inf and the new one finite; false if both -inf
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
          // PV of the previous chunk finished: P may be rewritten and O holds every PV so far
          // (an item's first chunk: the previous item's last PV was waited for at its end)
          if (!mbar_wait_warp(pv_done, (uint32_t)(gc - 1) & 1u, p.status)) {
            sm_ok = false;
            break;
          }
          tc_fence_after();
          if (rescale) {
#pragma unroll
            for (int part = 0; part < 4; ++part) {
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
            stmatrix_x4(smem_addr(Ps + sw128(mrow, 8 * hf + 2 * c + mchunk, kM)), pk[4 * c],
                        pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();  // P (generic stores) -> tensor-core reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (sm_ok && I.nloc > 0) sm_ok = mbar_wait_warp(pv_done, (uint32_t)(gc - 1) & 1u, p.status);
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
      if constexpr (kPersist) {
        // The item's end, among the 8 softmax warps only (named barrier 2): a failed wait in
        // any of them stops all of them at the same item, so none is left at a barrier.
        if (!sm_ok && lane == 0) *reinterpret_cast<volatile uint32_t*>(sm_abort) = 1u;
        asm volatile("bar.sync 2, %0;" ::"n"(32 * kSoftmaxWarps) : "memory");
        if (*reinterpret_cast<volatile uint32_t*>(sm_abort) != 0u) break;
        uint32_t o[32];
        float M0, M1, L0, L1;
        combine(I.nloc > 0, o, M0, M1, L0, L1);
        tc_fence_before();
        __syncwarp();
        if (I.nloc > 0 && lane == 0) mbar_arrive(o_free);  // the next item's PV may write O
        // every warp has read xml (and the abort word) before the next item writes them
        asm volatile("bar.sync 2, %0;" ::"n"(32 * kSoftmaxWarps) : "memory");
        if (early) pdl_wait();  // outputs are written only once the predecessor has completed
        store_out(I.tok, I.h_base, o, M0, M1, L0, L1);
      } else {
        break;  // one item
      }
    }
  }

  if constexpr (kPersist) {
    // every role is done with tensor memory and the pipeline buffers
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }

  __syncthreads();
  if (early) pdl_wait();  // outputs are written only once the predecessor has completed
  const int64_t tok = blockIdx.y;  // the CTA's one item
  const int h_base = (int)blockIdx.z * kM;
  const bool smx = warp < kSoftmaxWarps;
  uint32_t o[32];
  float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
  if (smx) combine(sm_ok && sm_nloc > 0, o, M0, M1, L0, L1);
  // Every role is done with tensor memory and the pipeline buffers.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }

  const int h0 = h_base + r0, h1 = h0 + 8;
  if (p.n_splits == 1) {
    if (smx) store_out(tok, h_base, o, M0, M1, L0, L1);
    return;
  }
  if (!p.cluster_merge) {
    if (smx) {
      const int64_t sbase = ((int64_t)split * p.tokens + tok) * p.H;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d0 = dc + 8 * i + 2 * tq;
        if (h0 < p.H)
          *reinterpret_cast<float2*>(p.ws_o + (sbase + h0) * kD + d0) =
              make_float2(f32(o[4 * i]), f32(o[4 * i + 1]));
        if (h1 < p.H)
          *reinterpret_cast<float2*>(p.ws_o + (sbase + h1) * kD + d0) =
              make_float2(f32(o[4 * i + 2]), f32(o[4 * i + 3]));
      }
      if (tq == 0 && hf == 0) {
        if (h0 < p.H) *reinterpret_cast<float2*>(p.ws_ml + (sbase + h0) * 2) = make_float2(M0, L0);
        if (h1 < p.H) *reinterpret_cast<float2*>(p.ws_ml + (sbase + h1) * 2) = make_float2(M1, L1);
      }
    }
    return;
  }
  // Cluster merge: park this split's partials in shared memory (the stage buffers are free).
  float* po = reinterpret_cast<float*>(KV);  // [64][kPStride]
  float* pml = po + kM * kPStride;           // [64][2]
  if (smx) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d0 = dc + 8 * i + 2 * tq;
      *reinterpret_cast<float2*>(po + r0 * kPStride + d0) =
          make_float2(f32(o[4 * i]), f32(o[4 * i + 1]));
      *reinterpret_cast<float2*>(po + (r0 + 8) * kPStride + d0) =
          make_float2(f32(o[4 * i + 2]), f32(o[4 * i + 3]));
    }
    if (tq == 0 && hf == 0) {
      *reinterpret_cast<float2*>(pml + r0 * 2) = make_float2(M0, L0);
      *reinterpret_cast<float2*>(pml + (r0 + 8) * 2) = make_float2(M1, L1);
    }
  }
  __syncthreads();
  cluster_sync();
  const int S = p.n_splits;
  const int rows_per = (kM + S - 1) / S;
  const int rb = split * rows_per, re = min(kM, rb + rows_per);
  constexpr int C4 = kD / 4;
  for (int x = threadIdx.x; x < (re - rb) * C4; x += kThreads) {
    const int row = rb + x / C4, c4 = x % C4;
    const int h = h_base + row;
    if (h >= p.H) continue;
    float2 ml[kMaxClusterSplits];
#pragma unroll
    for (int sp = 0; sp < kMaxClusterSplits; ++sp)
      ml[sp] = sp < S ? dsmem_ld_f32x2(pml + row * 2, sp) : make_float2(-INFINITY, 0.f);
    float Mx = -INFINITY;
#pragma unroll
    for (int sp = 0; sp < kMaxClusterSplits; ++sp) Mx = fmaxf(Mx, ml[sp].x);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float Lx = 0.f;
    if (Mx != -INFINITY) {
#pragma unroll
      for (int sp = 0; sp < kMaxClusterSplits; ++sp) {
        if (sp >= S || ml[sp].x == -INFINITY) continue;
        const float4 v = dsmem_ld_f32x4(po + row * kPStride + c4 * 4, sp);
        const float w = expf(ml[sp].x - Mx);
        Lx += w * ml[sp].y;
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
    }
    const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
    uint2 pk2;
    pk2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.out + (tok * p.H + h) * kD + c4 * 4) = pk2;
    if (p.lse != nullptr && c4 == 0) p.lse[tok * p.H + h] = Lx > 0.f ? Mx + logf(Lx) : -INFINITY;
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace

int attend_tc_chunk_keys() { return kKC; }

cudaError_t launch_attend_tc(const AttendArgs& a, int n_splits, int cluster, float* ws_o,
                             float* ws_ml, uint32_t* status, cudaStream_t stream) {
  TcParams prm;
  prm.q = a.q;
  prm.k_cmp = a.k_cmp;
  prm.v_cmp = a.v_cmp;
  prm.topk_idx = a.topk_idx;
  prm.topk_cnt = a.topk_cnt;
  prm.k_raw = a.k_raw;
  prm.v_raw = a.v_raw;
  prm.out = a.out;
  prm.lse = a.lse;
  prm.ws_o = ws_o;
  prm.ws_ml = ws_ml;
  prm.E = a.E;
  prm.N = a.N;
  prm.q_pos0 = a.q_pos0;
  prm.fresh_from = a.fresh_from;
  prm.block_table = a.paged ? a.paged->block_table : nullptr;
  prm.max_blocks = a.paged ? a.paged->max_blocks : 0;
  prm.n_pages = a.paged ? a.paged->n_pages : 0;
  prm.page_shift = 0;
  if (a.paged)
    while ((1 << prm.page_shift) < kPageTokens / a.m) ++prm.page_shift;
  prm.k = a.k;
  prm.m = a.m;
  prm.W = a.W;
  prm.Nq = a.Nq;
  prm.H = a.H;
  prm.n_splits = n_splits;
  prm.tokens = a.B * a.Nq;
  prm.sparse = a.topk_idx != nullptr;
  prm.cluster_merge = cluster;
  prm.status = status;
  // an unsplit launch (prefill) runs persistent CTAs, one per SM, over its (token, head group)
  // items
  const int groups = (a.H + kM - 1) / kM;
  const int64_t n_items = (int64_t)prm.tokens * groups;
  const bool persist = n_splits == 1 && !cluster;
  auto kern = persist ? attend_tc_kernel<true> : attend_tc_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  if (cluster && n_splits > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = persist ? dim3(1u, (unsigned)std::min<int64_t>(n_items, kNumSMs), 1u)
                        : dim3((unsigned)n_splits, (unsigned)prm.tokens, (unsigned)groups);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster ? (unsigned)n_splits : 1u;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cluster && n_splits > 8) {
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess || nclusters == 0) {
      (void)cudaGetLastError();
      return cudaErrorNotSupported;  // caller falls back to the workspace merge
    }
  }
  ProfScope prof(stream, prm.sparse ? "csa_attend" : "hca_attend");
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

}  // namespace csa
