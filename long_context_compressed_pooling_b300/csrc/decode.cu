// One CSA decode step in one launch: Lightning Indexer scores, the per-query top-k and the
// sparse attention over the selected entries plus the sliding window, for one query token per
// sequence.
//
// Lighthouse "deep deepseek v4 release" 八.3: CSA scores the compressed entries with the
// Lightning Indexer, keeps the top-k, and attends to the kept entries plus a sliding-window
// branch of raw tokens. 9fzt.com DeepSeek-V4 summary, item 4: the indexer's QK path runs in FP4
// and the selector works on scores rounded from FP32 to BF16.
//   s[j]  = bf16_rne( sum_h max(0, q_I,h . k_I,j) )                 visible entries j
//   S     = the min(k, visible) entries of largest s, ties to the lower index
//   out_h = softmax over {k_cmp[j] : j in S} + {k_raw[u] : u in window(t)} of q_h . key, times
//           the values
//
// One thread-block cluster of C CTAs per sequence (C chosen per launch, up to 16): CTA r scores
// the entries [r L, (r + 1) L) of the sequence and keeps their BF16 scores in shared memory, so
// no score leaves the chip. The cluster then selects through distributed shared memory and
// splits the selected entries and the window evenly for the attention, whose partial results it
// merges the same way. Phases:
//   1. indexer (the arithmetic of the decode path of indexer.cu): 4 loader warps stream 4-tile
//      slots of FP4 key codes and their UE8M0 scales with 16-byte cp.async into a 9-slot ring
//      (many small requests in flight per SM; one thread's bulk copies moved only ~30 GB/s per
//      SM here), starting before the other warps' set-up; an MMA warp issues one tcgen05
//      kind::mxf4 MMA per 128-entry tile (A = the tile read through the 32-byte swizzle, B = the
//      query's head blocks, each head in place and with its two 16-byte halves swapped, every
//      scale factor 1.0), 4 tiles per accumulator group; 8 epilogue warps apply the power-of-two
//      scales, take the ReLU sum over heads and round to BF16. Partial sums of e2m1 products are
//      exact in the fp32 accumulator and the scaled sums stay exact for the scale range of the
//      workloads, so the BF16 rounding is the only rounding.
//   2. top-k: the cluster's maximum, one histogram of (max - score) over the 255 BF16 steps
//      below it (per-warp histograms; an exact two-digit radix select when fewer than k scores
//      lie in that band), then each CTA counts its scores above / at the threshold and, from
//      every CTA's counts, writes its selected entries at their final ascending positions
//      (every thread owns a contiguous run of 8-key groups read with 16-byte loads).
//   3. attention (H <= 64 heads of dim 128 sharing one K/V head): the ordered key list (the
//      selected entries, then the window tokens) is cut into C equal runs; CTA r gathers its run
//      of K and V rows with cp.async into 128-byte-swizzled tiles (entry indices of other CTAs'
//      selections read through distributed shared memory), computes S = Q K^T (tcgen05 bf16,
//      M = 64 heads, N = up to 256 keys) into tensor memory, a one-pass softmax, O = P V into
//      tensor memory, and the cluster merges the C partial (max, sum, O) per head.
// Every wait on a copy, an MMA or another warp is bounded; on expiry the kernel records the
// timeout in the status word, stops using what it waited for, releases tensor memory and
// returns.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "prof.h"
#include "select.cuh"

namespace csa {
namespace {

constexpr int kLoadWarps = 4;    // warps 0-3: key copies (cp.async)
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kMmaWarp = 4;      // warp 4: tensor-memory allocation and every MMA
constexpr int kWorkWarp0 = 5;    // warps 5-12: indexer epilogue, then softmax
constexpr int kWorkWarps = 8;    // two per tensor-memory lane quarter (warp % 4)
constexpr int kWarps = kWorkWarp0 + kWorkWarps;
constexpr int kThreads = 32 * kWarps;
constexpr int kTileM = 128;      // entries per indexer tile
constexpr int kRowBytes = 32;    // d_I = 64 e2m1 codes
constexpr int kTileBytes = kTileM * kRowBytes;
constexpr int kSlotTiles = 4;   // one MMA group per slot
constexpr int kSlots = 9;       // 153 KB of key tiles in flight
constexpr int kSlotCodeBytes = kSlotTiles * kTileBytes;       // 16 KB
constexpr int kSlotBytes = kSlotCodeBytes + kSlotTiles * kTileM * 2;  // + UE8M0 scales
constexpr int kG = 4;            // tiles per MMA group
constexpr int kAcc = 4;          // accumulator groups (ring)
constexpr int kCols = 16;        // MMA N per tile: 4 heads x 2 blocks x (in place, swapped)
constexpr uint32_t kSfaCol = kAcc * kG * kCols;  // 256: scale factors (all 1.0)
constexpr uint32_t kSfbCol = kSfaCol + 16;
constexpr int kD = 128;          // head dim
constexpr int kM = 64;           // heads per CTA (MMA M)
constexpr uint32_t kOCol = 256;  // attention output accumulator, columns [256, 384)
constexpr int kQBytes = kM * kD * 2;                           // 16 KB
constexpr int kKVBytes = kDecodeMaxKeys * kD * 2;              // 64 KB per K or V tile
constexpr int kPBytes = kM * kDecodeMaxKeys * 2;               // 32 KB
constexpr int kUBytes = 2 * kKVBytes + kPBytes;                // 160 KB (phase 1 uses 136 KB)
static_assert(kSlots * kSlotBytes <= kUBytes, "ring fits the shared region");
constexpr int kPStride = kD + 4;                               // padded partial-output row
static_assert(kM * kPStride * 4 + kM * 8 <= kKVBytes, "partials fit the K tile");
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBins = 512;       // selection histogram: the BF16 score bits >> 6
constexpr int kSubBins = 64;     // inside the threshold bin: bits & 63
// merge inbox: [C][ceil(64 / C)][128] bf16 partial outputs, at most 79 head slots
constexpr int kMergeBf16 = 80 * kD;
static_assert(2048 * 2 + kMergeBf16 * 2 + 80 * 8 <= kDecodeMaxChunk * 2,
              "the merge inbox fits the score region");
static_assert(kThreads * 64 >= kDecodeMaxChunk, "a thread's segment fits a 64-bit mask");

// misc words
enum : int {
  kMiscMax = 0, kMiscGt, kMiscEq, kMiscBin, kMiscAbove, kMiscAboveLocal, kMiscAbort, kMiscTmem,
  kMiscCount = 16
};
constexpr int kNumBars = 2 * kSlots + 2 * kAcc + 4;
constexpr size_t kSmemBytes =
    1024 + kQBytes + kUBytes + kDecodeMaxChunk * 2 + 512 /*B operand*/ +
    (2 * kBins + kSubBins + kDecodeMaxCluster * (kSubBins + 1)) * 4 /*histograms*/ +
    kDecodeMaxKeys * 4 /*inbox*/ + 128 * 4 /*scan*/ + 2 * 32 * 4 /*cluster counts*/ +
    2 * 2 * kM * 4 /*row max / sum halves*/ + 8 * 4 /*row masks*/ + kMiscCount * 4 +
    kNumBars * 8 + 64;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct DecParams {
  const uint8_t* qi_codes;   // [B, H_I, 32]
  const uint8_t* qi_scales;  // [B, H_I, 2]
  const uint8_t* ki_codes;   // [B, E, 32]
  const uint8_t* ki_scales;  // [B, E, 2]
  uint16_t* scores;          // optional [B, E]
  int32_t* topk_idx;         // [B, k]
  int32_t* topk_cnt;         // [B]
  int64_t E, t;              // entries, query position
  int m, k, H_I, n_vis, chunk;
  int64_t keys_fresh_from;   // key tiles with an entry at or above it: copied after the wait
  int wait_first;            // grid-dependency wait before reading any input
  int split;                 // > 0: scores only, `split` CTAs per sequence without a cluster
  // attention (attend != 0)
  int attend, H, W, P;       // P: keys per CTA run
  const uint16_t* q;         // [B, H, 128]
  uint16_t* k_cmp;           // written only for the pooled entries
  uint16_t* v_cmp;           // [B, E, 128]
  const uint16_t* k_raw;
  const uint16_t* v_raw;     // [B, N, 128]
  uint16_t* out;             // [B, H, 128]
  float* lse;                // optional [B, H]
  int64_t N;
  // entries [pool_j0, pool_j1) of every sequence are pooled here from k_raw / v_raw / logits
  // (the blocks the step's tokens close), with csa_compress's arithmetic
  const float* logits;       // [B, N]
  int64_t pool_j0, pool_j1;
  uint32_t* status;
  long long wait_budget;
  uint32_t fault_mask;
};

// Byte offset of 16-byte chunk c (0..15) of row r in a 128-byte-swizzled K-major tile of R rows
// and 128 bf16 columns: two 64-column atoms of R x 128 B, chunk index XOR (row mod 8).
CSA_DEV uint32_t sw128(int r, int c, int R) {
  return (uint32_t)((c >> 3) * R * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

CSA_DEV void work_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }  // work warps
// the MMA warp and the work warps (the loaders never join the set-up)
CSA_DEV void setup_sync() {
  asm volatile("bar.sync 2, %0;" ::"n"(32 * (kWarps - kMmaWarp)) : "memory");
}

// Pools entries [p.pool_j0, p.pool_j1) of sequence b into k_cmp / v_cmp with the arithmetic of
// csa_compress (the same operations in the same order, so the entries are bit-identical):
// p_i = expf(w_i - max w) / sum, fp32 weighted sums, bf16 round-to-nearest-even. One warp; each
// half-warp an entry, each lane 8 of its 128 channels.
CSA_DEV void pool_entries(const DecParams& p, int64_t b, int lane) {
  const int64_t n = p.pool_j1 - p.pool_j0;
  const int c = lane & 15;
  for (int64_t e = lane >> 4; e < n; e += 2) {
    const int64_t j = p.pool_j0 + e;
    const int64_t tok0 = b * p.N + j * p.m;
    const float* wl = p.logits + tok0;
    float mx = -INFINITY;
    for (int i = 0; i < p.m; ++i) mx = fmaxf(mx, __ldg(wl + i));
    float acc_k[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float acc_v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float sum = 0.f;
    for (int i = 0; i < p.m; ++i) {
      const float pw = expf(__ldg(wl + i) - mx);
      sum += pw;
      acc8(acc_k, ldg_stream(p.k_raw + (tok0 + i) * kD + c * 8), pw);
      acc8(acc_v, ldg_stream(p.v_raw + (tok0 + i) * kD + c * 8), pw);
    }
    const float inv = 1.0f / sum;
    const int64_t o = (b * p.E + j) * kD + c * 8;
    *reinterpret_cast<uint4*>(p.k_cmp + o) = pack8(acc_k, inv);
    *reinterpret_cast<uint4*>(p.v_cmp + o) = pack8(acc_v, inv);
  }
}

__global__ void __launch_bounds__(kThreads, 1) csa_decode_kernel(const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* Qs = base;                                     // [2 atoms][64 rows][128 B]
  uint8_t* U = Qs + kQBytes;                              // ring, then K | V | P tiles
  uint16_t* keys = reinterpret_cast<uint16_t*>(U + kUBytes);       // [chunk] BF16 scores
  uint8_t* btile = reinterpret_cast<uint8_t*>(keys + kDecodeMaxChunk);  // 16 rows x 32 B
  uint32_t* hist = reinterpret_cast<uint32_t*>(btile + 512);  // [512] this CTA: bits >> 6
  uint32_t* sub = hist + kBins;      // [64] this CTA: the threshold bin by bits & 63
  uint32_t* gall = sub + kSubBins;   // [512] the cluster's histogram (every CTA adds into it)
  uint32_t* subs = gall + kBins;     // [16][64] every CTA's threshold-bin counts (pushed)
  uint32_t* cab = subs + kDecodeMaxCluster * kSubBins;  // [16] every CTA's count above the bin
  int32_t* inbox = reinterpret_cast<int32_t*>(cab + kDecodeMaxCluster);  // [256] run entries
  uint32_t* gsum = reinterpret_cast<uint32_t*>(inbox + kDecodeMaxKeys);  // scan scratch [128]
  uint32_t* cgt = gsum + 128;        // [32] every CTA's count above the threshold
  uint32_t* ceq = cgt + 32;          // [32] ... equal to it
  float* xm = reinterpret_cast<float*>(ceq + 32);  // [2 halves][64 rows] softmax row maxima
  float* xs = xm + 2 * kM;                          // [2 halves][64 rows] row sums
  uint32_t* rowmask = reinterpret_cast<uint32_t*>(xs + 2 * kM);  // [8] valid attention keys
  uint32_t* misc = rowmask + 8;
  uint64_t* bars = reinterpret_cast<uint64_t*>(misc + kMiscCount);
  uint64_t* full = bars;                    // [kSlots] key copies landed (loader threads)
  uint64_t* empty = full + kSlots;          // [kSlots] MMAs and epilogue done with a slot
  uint64_t* tfull = empty + kSlots;         // [kAcc] accumulator group written
  uint64_t* tempty = tfull + kAcc;          // [kAcc] accumulator group read
  uint64_t* drain = tempty + kAcc;          // every indexer MMA finished
  uint64_t* s_full = drain + 1;             // QK^T finished
  uint64_t* p_full = s_full + 1;            // P written (8 warps)
  uint64_t* o_full = p_full + 1;            // PV finished
  // the runs' partial outputs for the heads this CTA merges, pushed by every CTA (bf16,
  // normalised by the run's own sum), and each run's (maximum, sum) per head: they land in the
  // score region, which is dead once the selection is written
  uint16_t* pin = keys + 2048;                                   // [16][hp][128] bf16
  float2* pinml = reinterpret_cast<float2*>(keys + 2048 + kMergeBf16);  // [16][hp]

  // scores only (split > 0): no cluster, CTA blockIdx.x % split of its sequence
  const bool score_only = p.split > 0;
  const uint32_t C = score_only ? (uint32_t)p.split : cluster_nctarank();
  const uint32_t rank = score_only ? blockIdx.x % (uint32_t)p.split : cluster_ctarank();
  const int64_t b = blockIdx.x / C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const long long budget = p.wait_budget;

  pdl_trigger();
  if (p.wait_first) pdl_wait();

  const int n = p.n_vis;
  const bool select_all = n <= p.k;  // every visible entry is selected: no selection to make
  const int cnt = min(p.k, n);
  const int lo = min(n, (int)rank * p.chunk);
  const int len = min(n, lo + p.chunk) - lo;
  // the scores are computed unless every entry is selected and no score output is requested
  const int ntiles = (select_all && p.scores == nullptr) ? 0 : (len + kTileM - 1) / kTileM;
  const int nunits = (ntiles + kSlotTiles - 1) / kSlotTiles;
  const int ngroups = (ntiles + kG - 1) / kG;
  const int64_t w0 = p.t - p.W + 1 > 0 ? p.t - p.W + 1 : 0;
  const int nw = p.W > 0 ? (int)(p.t - w0 + 1) : 0;
  const int n_keys = cnt + nw;

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], kLoadThreads);
      mbar_init(&empty[s], 1 + kWorkWarps);
    }
    for (int a = 0; a < kAcc; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kWorkWarps);
    }
    mbar_init(drain, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, kWorkWarps);
    mbar_init(o_full, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < kMiscCount; i += kThreads) misc[i] = 0u;
  for (int i = tid; i < kBins + kSubBins + kBins + kDecodeMaxCluster * (kSubBins + 1); i += kThreads)
    hist[i] = 0u;  // hist, sub, gall, subs, cab
  __syncthreads();  // barriers initialised, misc words and histograms cleared
  // The other CTAs add into gall / store into subs, cab and inbox once they pass the matching
  // wait below: this arrive orders the clearing before it.
  if (!score_only) cluster_arrive();

  bool ok = true;  // this thread's waits all succeeded (a timeout stops the phases after it)
  float qsc[8];  // query scale of (head, block), 2^(e - 127) (work warps; loaded during set-up)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = i >> 1;
    const uint32_t e = warp >= kWorkWarp0 && h < p.H_I ? p.qi_scales[(b * p.H_I + h) * 2 + (i & 1)]
                                                      : 127u;
    qsc[i] = exp2_int((int)e - 127);
  }
  if (warp < kLoadWarps) {
    // ======== loaders: the key codes and scales of this CTA's chunk, slot by slot ========
    // Every loader thread copies 16-byte pieces with cp.async and arrives on the slot's barrier
    // when its own copies have landed; nothing here waits for the set-up of the other warps.
    // Key tiles below keys_fresh_from cannot be written by the kernel this one overlaps, so
    // they are copied at once; the first slot holding a later entry waits for that kernel.
    const int lt = tid;  // 0 .. kLoadThreads - 1
    bool waited = p.wait_first != 0;
    const bool skip = (p.fault_mask & kFaultSkipKeyCopies) != 0;
    for (int u = 0; u < nunits && !skip; ++u) {
      const int slot = u % kSlots;
      if (u >= kSlots &&
          !mbar_wait_warp(&empty[slot], (uint32_t)((u / kSlots) - 1) & 1u, p.status, budget)) {
        ok = false;
        break;
      }
      const int r0 = u * kSlotTiles * kTileM;
      if (!waited && (int64_t)lo + r0 + kSlotTiles * kTileM > p.keys_fresh_from) {
        pdl_wait();
        waited = true;
      }
      int rows = min(len - r0, kSlotTiles * kTileM);
      rows = (rows + 7) & ~7;  // whole 16-byte runs of scales; E % 8 == 0 keeps them inside
      uint8_t* sb = U + slot * kSlotBytes;
      const uint8_t* gc = p.ki_codes + (b * p.E + lo + r0) * kRowBytes;
      const uint8_t* gs = p.ki_scales + (b * p.E + lo + r0) * 2;
      const int code_chunks = rows * (kRowBytes / 16), scale_chunks = rows / 8;
      for (int x = lt; x < code_chunks; x += kLoadThreads)
        cp_async_16(sb + x * 16, gc + x * 16, 16u);
      for (int x = lt; x < scale_chunks; x += kLoadThreads)
        cp_async_16(sb + kSlotCodeBytes + x * 16, gs + x * 16, 16u);
      cp_async_mbar_arrive_noinc(&full[slot]);
    }
    cp_async_wait<0>();  // never leave with copies in flight
  } else {
    // ======== set-up of the MMA and work warps (the loaders are already copying) ========
    // the attention's queries (an input of the call) start arriving at once
    if (p.attend) {
      for (int x = tid - kLoadThreads; x < kM * 16; x += kThreads - kLoadThreads) {
        const int r = x >> 4, c = x & 15;
        const bool in = r < p.H;
        cp_async_16(Qs + sw128(r, c, kM), in ? p.q + (b * p.H + r) * kD + c * 8 : p.q,
                    in ? 16u : 0u);
      }
      cp_async_commit();
    }
    // B operand of the indexer: row r = head r / 4, block r % 2, halves swapped when
    // (r / 2) % 2; every row holds one 16-byte block of the head and zeros, stored through the
    // 32-byte swizzle
    for (int x = tid - kLoadThreads; x < 32; x += kThreads - kLoadThreads) {
      const int r = x >> 1, c = x & 1;
      const int h = r >> 2, sw = (r >> 1) & 1, blk = r & 1;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (h < p.H_I && c == (blk ^ sw))
        v = *reinterpret_cast<const uint4*>(p.qi_codes + (b * p.H_I + h) * 32 + blk * 16);
      *reinterpret_cast<uint4*>(btile + r * kRowBytes + ((c ^ ((r >> 2) & 1)) << 4)) = v;
    }
    fence_proxy_async_smem();
    if (warp == kMmaWarp) {
      tmem_alloc(reinterpret_cast<uint32_t*>(&misc[kMiscTmem]), 512);
      tmem_relinquish();
    }
    __syncwarp();
    tc_fence_before();
    setup_sync();
    tc_fence_after();
  }
  const uint32_t tmem = misc[kMiscTmem];  // read by the MMA and work warps after setup_sync
  if (warp >= kWorkWarp0) {
    if (warp < kWorkWarp0 + 4) {  // scale factors 1.0 for A and B, lane quarter warp % 4
      const uint32_t lb = (uint32_t)((warp & 3) * 32) << 16;
#pragma unroll
      for (int c = 0; c < 32; c += 8) tmem_st8_fill(tmem + lb + kSfaCol + c, 0x7F7F7F7Fu);
      tmem_st_wait();
    }
  }
  if (warp >= kMmaWarp) {
    __syncwarp();
    tc_fence_before();
    setup_sync();
    tc_fence_after();
  }

  // The blocks this step closes: pooled by one warp of the cluster's last CTA, before its
  // epilogue work; the attention reads them only after the cluster barriers below.
  if (p.pool_j1 > p.pool_j0 && rank == C - 1 && warp == kWarps - 1) {
    pdl_wait();  // the entries it writes may still be read by the kernel before this one
    pool_entries(p, b, lane);
  }

  // ======================= phase 1: indexer scores into shared memory =======================
  if (ntiles > 0 && warp == kMmaWarp) {
    const uint32_t idesc = idesc_mxf4(kTileM, kCols);
    const uint64_t bdesc = smem_desc(smem_addr(btile), 16, 256, kSwizzle32B);
    for (int g = 0; g < ngroups; ++g) {
      const int a = g % kAcc;
      const int u = g * kG / kSlotTiles, slot = u % kSlots;
      if (!mbar_wait_warp(&tempty[a], ((uint32_t)(g / kAcc) & 1u) ^ 1u, p.status, budget) ||
          !mbar_wait_warp(&full[slot], (uint32_t)(u / kSlots) & 1u, p.status, budget)) {
        ok = false;
        break;
      }
      fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor-core reads
      tc_fence_after();
      const int nt = min(kG, ntiles - g * kG);
      const bool unit_done = (g + 1) * kG >= min(ntiles, (u + 1) * kSlotTiles);
      if (elect_one()) {
        for (int i = 0; i < nt; ++i) {
          const int it = g * kG + i;
          const uint64_t adesc = smem_desc(
              smem_addr(U + slot * kSlotBytes + (it % kSlotTiles) * kTileBytes), 16, 256,
              kSwizzle32B);
          umma_mxf4(tmem + (uint32_t)(a * kG * kCols + i * kCols), adesc, bdesc, idesc,
                    tmem + kSfaCol, tmem + kSfbCol, 0u);
        }
        if (unit_done) umma_commit(&empty[slot]);
        umma_commit(&tfull[a]);
      }
      __syncwarp();
    }
    if (elect_one()) umma_commit(drain);  // arrives once every MMA issued above has finished
    __syncwarp();
    if (!mbar_wait_warp(drain, 0, p.status, budget)) ok = false;
  } else if (ntiles > 0 && warp >= kWorkWarp0) {
    // epilogue: warp (quarter q, sub) reads tiles i % 2 == sub of each group
    const int q = warp & 3, sub = (warp - kWorkWarp0) >> 2;
    const int row = q * 32 + lane;
    const bool swapped = ((row >> 2) & 1) != 0;  // unswizzled row read through the swizzle
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    for (int g = 0; g < ngroups; ++g) {
      const int a = g % kAcc;
      const int u = g * kG / kSlotTiles, slot = u % kSlots;
      if (!mbar_wait_warp(&tfull[a], (uint32_t)(g / kAcc) & 1u, p.status, budget) ||
          !mbar_wait_warp(&full[slot], (uint32_t)(u / kSlots) & 1u, p.status, budget)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool unit_done = (g + 1) * kG >= min(ntiles, (u + 1) * kSlotTiles);
      uint32_t r[2][16];
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int i = sub + 2 * x;
        if (g * kG + i < ntiles)
          tmem_ld16(tmem + lb + (uint32_t)(a * kG * kCols + i * kCols), r[x]);
      }
      tmem_ld_wait();
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int it = g * kG + sub + 2 * x;
        const int jl = it * kTileM + row;  // entry index within the chunk
        if (it >= ntiles || jl >= len) continue;
        const uint32_t sbits = *reinterpret_cast<const uint16_t*>(
            U + slot * kSlotBytes + kSlotCodeBytes + ((it % kSlotTiles) * kTileM + row) * 2);
        const float sk0 = exp2_int((int)(sbits & 0xFF) - 127);
        const float sk1 = exp2_int((int)(sbits >> 8) - 127);
        float sc = 0.f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          // the two block partial sums of head h, from the column pair matching this row
          const float d0 = __uint_as_float(swapped ? r[x][4 * h + 2] : r[x][4 * h]);
          const float d1 = __uint_as_float(swapped ? r[x][4 * h + 3] : r[x][4 * h + 1]);
          float dot = fmaf(d0 * qsc[2 * h], sk0, 0.f);
          dot = fmaf(d1 * qsc[2 * h + 1], sk1, dot);
          sc += fmaxf(dot, 0.f);  // rows of absent heads are zero
        }
        sc += 0.0f;  // -0 -> +0
        const uint16_t bits = f32_to_bf16_bits(sc);
        keys[jl] = bits;
        if (!select_all && !score_only) atomicAdd(&hist[bits >> 6], 1u);  // 64-step bins
        if (p.scores) p.scores[b * p.E + lo + jl] = bits;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[a]);
        if (unit_done) mbar_arrive(&empty[slot]);
      }
    }
  }
  if (!ok) misc[kMiscAbort] = 1u;  // benign race: every writer stores 1
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // A timeout anywhere in the cluster must not leave the other CTAs waiting at a cluster
  // barrier: every CTA still passes every barrier below, skipping the work.
  const bool aborted = misc[kMiscAbort] != 0u;
  if (score_only) {  // the scores are written: release tensor memory and leave
    pdl_wait();      // completion stays ordered after the predecessor's
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
    return;
  }

  // ======================= phase 2: top-k through the cluster =======================
  // The threshold T (the k-th largest score) in two cluster rounds, every exchange a store or
  // atomic add into the other CTAs' shared memory: (A) each CTA adds its histogram of the
  // scores' bits >> 6 (built by the epilogue) into every CTA's copy of the cluster histogram,
  // which gives the bin holding T; (B) each CTA sends its counts of scores in that bin by their
  // 6 low bits, and above it, to every CTA, which gives T, how many scores equal to T are
  // taken, and every CTA's counts above / at T. BF16 scores are non-negative here, so their bit
  // patterns order like their values. Each CTA then writes its selected entries at their final
  // ascending positions and, for the attention, sends each to the CTA whose run holds it.
  cluster_wait();  // every CTA has cleared its exchange buffers
  uint32_t T = 0, need_eq = 0;
  // this thread's contiguous segment of the chunk: a multiple of 8 keys (16-byte loads), at
  // most 64 (kThreads * 64 >= kDecodeMaxChunk), so its selection fits 64-bit masks
  const int seg = ((len + kThreads - 1) / kThreads + 7) & ~7;
  const int s0 = min(len, tid * seg), s1 = min(len, s0 + seg);
  if (!select_all) {
    for (int q = tid; q < kBins; q += kThreads) {
      const uint32_t v = hist[q];
      if (v != 0u)
        for (uint32_t c = 0; c < C; ++c) dsmem_red_add_u32(dsmem_map(&gall[q], c), v);
    }
    cluster_sync();  // (A) the cluster histogram is complete in every CTA
    if (warp == 0) {  // lane l holds bins [496 - 16 l, 512 - 16 l), counted from the top
      uint32_t loc = 0;
#pragma unroll
      for (int j = 0; j < 16; ++j) loc += gall[kBins - 1 - 16 * lane - j];
      uint32_t inc = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      const uint32_t need = (uint32_t)p.k;
      uint32_t run = inc - loc;
      if (run < need && need <= inc) {
        for (int j = 0; j < 16; ++j) {
          const int bin = kBins - 1 - 16 * lane - j;
          if (run + gall[bin] >= need) {
            misc[kMiscBin] = (uint32_t)bin;
            misc[kMiscAbove] = run;  // scores in bins above it, cluster-wide
            break;
          }
          run += gall[bin];
        }
      }
    }
    __syncthreads();
    const uint32_t bstar = misc[kMiscBin], above_g = misc[kMiscAbove];
    // this CTA's scores above bstar, and its scores inside bstar by their 6 low bits; the
    // thread's keys above / inside bstar as bit masks
    uint64_t m_hi = 0, m_in = 0;
    for (int r = s0; r < s1; r += 8) {
      const uint4 v = *reinterpret_cast<const uint4*>(keys + r);
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t kk = (w4[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
        if (r + e < s1) {
          const uint64_t bit = 1ull << (r + e - s0);
          if ((kk >> 6) > bstar) m_hi |= bit;
          if ((kk >> 6) == bstar) {
            m_in |= bit;
            atomicAdd(&sub[kk & 63u], 1u);
          }
        }
      }
    }
    {
      uint32_t a_loc = (uint32_t)__popcll(m_hi);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a_loc += __shfl_xor_sync(0xffffffffu, a_loc, o);
      if (lane == 0 && a_loc) atomicAdd(&misc[kMiscAboveLocal], a_loc);
    }
    __syncthreads();
    constexpr int kSubChunks = kSubBins / 4;  // 16-byte pieces of the counts
    for (int x = tid; x < (int)C * (kSubChunks + 1); x += kThreads) {
      const uint32_t c = (uint32_t)(x / (kSubChunks + 1)), j = (uint32_t)(x % (kSubChunks + 1));
      if (j < (uint32_t)kSubChunks)
        dsmem_st_u32x4(dsmem_map(&subs[rank * kSubBins + 4 * j], c),
                       *reinterpret_cast<const uint4*>(&sub[4 * j]));
      else
        dsmem_st_u32(dsmem_map(&cab[rank], c), misc[kMiscAboveLocal]);
    }
    cluster_sync();  // (B) every CTA's threshold-bin counts are in every CTA
    if (warp == 0) {
      // lane l: the cluster's counts of scores bstar * 64 + {2l, 2l + 1}; T from the top
      uint32_t c_lo = 0, c_hi = 0;
      for (uint32_t c = 0; c < C; ++c) {
        c_lo += subs[c * kSubBins + 2 * lane];
        c_hi += subs[c * kSubBins + 2 * lane + 1];
      }
      const uint32_t need = (uint32_t)p.k - above_g;
      const uint32_t loc = c_lo + c_hi;
      uint32_t inc = loc;  // inclusive count from the top (lane 31 holds the largest scores)
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, inc, o);
        if (lane + o < 32) inc += v;
      }
      const uint32_t exc = inc - loc;  // scores in higher lanes' bins
      // the k-th score is in this lane's upper bin, or in its lower one
      const bool in_hi = exc < need && need <= exc + c_hi;
      const bool in_lo = exc + c_hi < need && need <= inc;
      const uint32_t hit = __ballot_sync(0xffffffffu, in_hi || in_lo);
      const int hl = __ffs(hit) - 1;
      const int ts = 2 * hl + (__shfl_sync(0xffffffffu, in_hi ? 1 : 0, hl) ? 1 : 0);
      const uint32_t before = __shfl_sync(0xffffffffu, in_hi ? exc : exc + c_hi, hl);
      if (lane < (int)C) {  // CTA `lane`: scores above T and equal to T
        uint32_t gt = cab[lane];
        for (int s2 = ts + 1; s2 < kSubBins; ++s2) gt += subs[lane * kSubBins + s2];
        cgt[lane] = gt;
        ceq[lane] = subs[lane * kSubBins + ts];
      }
      if (lane == 0) {
        misc[kMiscBin] = (bstar << 6) | (uint32_t)ts;
        misc[kMiscAbove] = need - before;  // scores equal to T that are taken
      }
    }
    __syncthreads();
    T = misc[kMiscBin];
    need_eq = misc[kMiscAbove];
    // the thread's keys above / at T (those inside bstar compared one by one)
    uint64_t m_gt = m_hi, m_eq = 0;
    for (uint64_t m = m_in; m != 0; m &= m - 1) {
      const int i = __ffsll((long long)m) - 1;
      const uint32_t kk = keys[s0 + i];
      if (kk > T) m_gt |= 1ull << i;
      if (kk == T) m_eq |= 1ull << i;
    }
    uint32_t ex_gt, ex_eq, tot_gt, tot_eq;
    block_scan2((uint32_t)__popcll(m_gt), (uint32_t)__popcll(m_eq), &ex_gt, &ex_eq, &tot_gt,
                &tot_eq, gsum, gsum + 64);
    uint32_t gb = ex_gt, eb = ex_eq;  // keys above / at T before this thread's segment
    for (uint32_t c = 0; c < rank; ++c) {
      gb += cgt[c];
      eb += ceq[c];
    }
    int32_t* out_idx = p.topk_idx + b * p.k;
    if (!aborted) {
      for (uint64_t m = m_gt | m_eq; m != 0; m &= m - 1) {
        const int i = __ffsll((long long)m) - 1;
        const uint64_t below = (1ull << i) - 1;
        const uint32_t g_b = gb + (uint32_t)__popcll(m_gt & below);
        const uint32_t e_b = eb + (uint32_t)__popcll(m_eq & below);
        int pos = -1;
        if ((m_gt >> i) & 1ull)
          pos = (int)(g_b + min(e_b, need_eq));
        else if (e_b < need_eq)
          pos = (int)(g_b + e_b);
        if (pos >= 0 && pos < p.k) {
          const int j = lo + s0 + i;
          out_idx[pos] = j;
          if (p.attend) {  // to the CTA whose attention run holds position pos
            const uint32_t dst = (uint32_t)(pos / p.P);
            dsmem_st_u32(dsmem_map(&inbox[pos - (int)dst * p.P], dst), (uint32_t)j);
          }
        }
      }
    }
    if (rank == 0 && tid == 0) p.topk_cnt[b] = cnt;
  } else {
    for (int r = (int)rank * kThreads + tid; r < p.k; r += (int)C * kThreads)
      p.topk_idx[b * p.k + r] = r < n ? r : -1;
    if (rank == 0 && tid == 0) p.topk_cnt[b] = cnt;
  }

  // ======================= phase 3: attention over this CTA's run of keys =======================
  if (p.attend) {
    __syncthreads();
    cluster_sync();  // (C) every run's selected entries are in its CTA's inbox
    pdl_wait();      // the entry cache may be the output of the kernel before this one
    const int p0 = min(n_keys, (int)rank * p.P);
    const int nk = aborted ? 0 : min(n_keys, p0 + p.P) - p0;
    const int nkp = (nk + 15) & ~15;  // MMA N (a multiple of 16), keys [nk, nkp) are masked
    uint8_t* Kt = U;
    uint8_t* Vt = U + kKVBytes;
    uint8_t* Pt = U + 2 * kKVBytes;
    int64_t* rowsrc = reinterpret_cast<int64_t*>(keys);  // the scores are no longer needed
    static_assert(kDecodeMaxKeys * 8 <= 2048 * 2, "row sources stay below the merge inbox");
    constexpr long long kRawBit = 1LL << 62;
    // source row of every key of the run: entry (element offset into k_cmp / v_cmp) or raw
    // window token (bit 62); -1 = none (zero-filled, masked)
    for (int i = tid; i < nkp; i += kThreads) {
      long long src = -1;
      if (i < nk) {
        const int pp = p0 + i;
        if (pp < cnt) {
          const int64_t j = select_all ? (int64_t)pp : (int64_t)inbox[i];
          if (j < 0 || j >= p.E)
            atomicOr(p.status, kFlagBadIndex);
          else
            src = (b * p.E + j) * kD;
        } else {
          src = ((b * p.N + w0 + (pp - cnt)) * kD) | kRawBit;
        }
      }
      rowsrc[i] = src;
    }
    if (tid < 8) rowmask[tid] = 0u;
    bool my_bad = false;
    for (int i = tid; i < nk; i += kThreads) my_bad |= rowsrc[i] < 0;
    // every key of the run has a row (no bad index): the softmax masks by position alone
    const bool any_bad = __syncthreads_or(my_bad) != 0;
    for (int i = tid; i < nkp; i += kThreads)
      if (rowsrc[i] >= 0) atomicOr(&rowmask[i >> 5], 1u << (i & 31));
    for (int x = tid; x < nkp * 16; x += kThreads) {
      const int i = x >> 4, c = x & 15;
      const long long src = rowsrc[i];
      const bool valid = src >= 0;
      const bool raw = (src & kRawBit) != 0;
      const int64_t e = src & (kRawBit - 1);
      const uint16_t* ks = valid ? (raw ? p.k_raw : p.k_cmp) + e + c * 8 : p.k_raw;
      const uint16_t* vs = valid ? (raw ? p.v_raw : p.v_cmp) + e + c * 8 : p.v_raw;
      const uint32_t off = sw128(i, c, kDecodeMaxKeys);
      cp_async_16(Kt + off, ks, valid ? 16u : 0u);
      cp_async_16(Vt + off, vs, valid ? 16u : 0u);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
    const int q = warp & 3, hf = (warp - kWorkWarp0) >> 2;
    const int g = lane >> 2, tq = lane & 3;
    const int r0 = q * 16 + g;  // this thread's rows r0 and r0 + 8 (work warps)
    const uint32_t lb = (uint32_t)(q * 32) << 16;
    bool att_ok = true;
    if (nk > 0) {
      if (warp == kMmaWarp) {
        // S = Q K^T: M = 64 heads, N = nkp keys, K = 128 in 8 steps of 16
        const uint32_t id_qk = idesc_bf16(kM, nkp, false, false);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t atom = kk >> 2, kin = (kk & 3) * 32;
            const uint64_t ad =
                smem_desc(smem_addr(Qs) + atom * kM * 128 + kin, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(smem_addr(Kt) + atom * kDecodeMaxKeys * 128 + kin, 16,
                                          1024, kSwizzle128B);
            umma_bf16(tmem, ad, bd, id_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
        }
        __syncwarp();
        // O = P V: M = 64, N = 128, K = nkp keys in steps of 16
        if (!mbar_wait_warp(p_full, 0, p.status, budget)) {
          att_ok = false;
        } else {
          tc_fence_after();
          const uint32_t id_pv = idesc_bf16(kM, kD, false, true);
          if (elect_one()) {
            for (int kk = 0; kk < nkp / 16; ++kk) {
              const uint32_t atom = kk >> 2, kin = (kk & 3) * 32;
              const uint64_t ad =
                  smem_desc(smem_addr(Pt) + atom * kM * 128 + kin, 16, 1024, kSwizzle128B);
              // V rows are keys (the K dimension), d contiguous: MN-major B, 64-column atoms
              // kDecodeMaxKeys * 128 bytes apart, 8-key groups 1024 bytes apart
              const uint64_t bd = smem_desc(smem_addr(Vt) + kk * 16 * 128, kDecodeMaxKeys * 128,
                                            1024, kSwizzle128B);
              umma_bf16(tmem + kOCol, ad, bd, id_pv, kk > 0 ? 1u : 0u);
            }
            umma_commit(o_full);
          }
          __syncwarp();
          // tensor memory is freed only after the MMAs finished
          if (!mbar_wait_warp(o_full, 0, p.status, budget)) att_ok = false;
        }
      } else if (warp >= kWorkWarp0) {
        // softmax: warp (q, hf) holds rows 16q .. 16q + 15, key columns [hf nkp/2, (hf+1) nkp/2),
        // one 8-column group per tensor-memory load (a short loop body): the masked row maxima
        // first, then the probabilities (re-read) written to P as bf16
        const int half = nkp >> 1;  // a multiple of 8
        const int c0 = hf * half;
        if (!mbar_wait_warp(s_full, 0, p.status, budget)) att_ok = false;
        tc_fence_after();
        float mx0 = -INFINITY, mx1 = -INFINITY;
        for (int g8 = c0; g8 < c0 + half && att_ok; g8 += 8) {
          uint32_t t4[4];
          tmem_ld_16x256b_x1(tmem + lb + (uint32_t)g8, t4);
          tmem_ld_wait();
          const int col = g8 + 2 * tq;  // and col + 1
          const bool v0 = col < nk && (!any_bad || ((rowmask[col >> 5] >> (col & 31)) & 1u));
          const bool v1 =
              col + 1 < nk && (!any_bad || ((rowmask[(col + 1) >> 5] >> ((col + 1) & 31)) & 1u));
          if (v0) {
            mx0 = fmaxf(mx0, __uint_as_float(t4[0]));
            mx1 = fmaxf(mx1, __uint_as_float(t4[2]));
          }
          if (v1) {
            mx0 = fmaxf(mx0, __uint_as_float(t4[1]));
            mx1 = fmaxf(mx1, __uint_as_float(t4[3]));
          }
        }
#pragma unroll
        for (int x = 1; x < 4; x <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
        }
        if (tq == 0) {
          xm[hf * kM + r0] = mx0;
          xm[hf * kM + r0 + 8] = mx1;
        }
        work_sync();
        M0 = fmaxf(xm[r0], xm[kM + r0]);
        M1 = fmaxf(xm[r0 + 8], xm[kM + r0 + 8]);
        const float nb0 = M0 == -INFINITY ? 0.f : -M0 * kLog2e;
        const float nb1 = M1 == -INFINITY ? 0.f : -M1 * kLog2e;
        float s0 = 0.f, s1 = 0.f;
        for (int g8 = c0; g8 < c0 + half; g8 += 8) {
          uint32_t t4[4] = {0u, 0u, 0u, 0u};
          if (att_ok) {
            tmem_ld_16x256b_x1(tmem + lb + (uint32_t)g8, t4);
            tmem_ld_wait();
          }
          const int col = g8 + 2 * tq;
          const bool v0 = att_ok && col < nk &&
                          (!any_bad || ((rowmask[col >> 5] >> (col & 31)) & 1u));
          const bool v1 = att_ok && col + 1 < nk &&
                          (!any_bad || ((rowmask[(col + 1) >> 5] >> ((col + 1) & 31)) & 1u));
          const float p00 = v0 ? ex2_approx(fmaf(__uint_as_float(t4[0]), kLog2e, nb0)) : 0.f;
          const float p01 = v1 ? ex2_approx(fmaf(__uint_as_float(t4[1]), kLog2e, nb0)) : 0.f;
          const float p10 = v0 ? ex2_approx(fmaf(__uint_as_float(t4[2]), kLog2e, nb1)) : 0.f;
          const float p11 = v1 ? ex2_approx(fmaf(__uint_as_float(t4[3]), kLog2e, nb1)) : 0.f;
          s0 += p00 + p01;
          s1 += p10 + p11;
          // P[row][key] bf16, K-major over keys: atom key / 64, 16-byte chunk (key % 64) / 8
          const int atom = g8 >> 6, ch = (g8 & 63) >> 3;
          uint8_t* pa = Pt + atom * kM * 128;
          *reinterpret_cast<uint32_t*>(pa + r0 * 128 + ((ch ^ (r0 & 7)) << 4) + tq * 4) =
              pack_bf16x2(p00, p01);
          *reinterpret_cast<uint32_t*>(pa + (r0 + 8) * 128 + ((ch ^ ((r0 + 8) & 7)) << 4) +
                                       tq * 4) = pack_bf16x2(p10, p11);
        }
#pragma unroll
        for (int x = 1; x < 4; x <<= 1) {
          s0 += __shfl_xor_sync(0xffffffffu, s0, x);
          s1 += __shfl_xor_sync(0xffffffffu, s1, x);
        }
        if (tq == 0) {
          xs[hf * kM + r0] = s0;
          xs[hf * kM + r0 + 8] = s1;
        }
        fence_proxy_async_smem();  // P (generic stores) -> tensor-core reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        work_sync();
        L0 = xs[r0] + xs[kM + r0];
        L1 = xs[r0 + 8] + xs[kM + r0 + 8];
      }
    }
    // This run's partial output of every head, normalised by the run's own sum and rounded to
    // bf16, goes with its (maximum, sum) to the CTA that merges that head.
    const int hp = (kM + (int)C - 1) / (int)C;  // heads merged per CTA
    if (warp >= kWorkWarp0) {
      const int dc = hf * 64;
      uint32_t o[32];
#pragma unroll
      for (int x = 0; x < 32; ++x) o[x] = 0u;
      if (nk > 0 && att_ok) {
        if (mbar_wait_warp(o_full, 0, p.status, budget)) {
          tc_fence_after();
          tmem_ld_16x256b_x8(tmem + lb + kOCol + (uint32_t)dc, o);
          tmem_ld_wait();
        } else {
          att_ok = false;
        }
      }
      if (!att_ok) {
        M0 = M1 = -INFINITY;
        L0 = L1 = 0.f;
      }
      const float i0 = L0 > 0.f ? 1.f / L0 : 0.f, i1 = L1 > 0.f ? 1.f / L1 : 0.f;
      // staged row-major in the dead K tile, then sent in 16-byte pieces
      uint16_t* stage = reinterpret_cast<uint16_t*>(Kt);  // [64][128] bf16
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d0 = dc + 8 * i + 2 * tq;
        *reinterpret_cast<uint32_t*>(&stage[r0 * kD + d0]) =
            pack_bf16x2(__uint_as_float(o[4 * i]) * i0, __uint_as_float(o[4 * i + 1]) * i0);
        *reinterpret_cast<uint32_t*>(&stage[(r0 + 8) * kD + d0]) =
            pack_bf16x2(__uint_as_float(o[4 * i + 2]) * i1, __uint_as_float(o[4 * i + 3]) * i1);
      }
      if (tq == 0 && hf == 0) {
        for (int rr = 0; rr < 2; ++rr) {
          const int h = r0 + 8 * rr;
          const uint32_t dst = (uint32_t)(h / hp);
          dsmem_st_f32x2(dsmem_map(&pinml[(int)rank * hp + (h - (int)dst * hp)], dst),
                         rr ? make_float2(M1, L1) : make_float2(M0, L0));
        }
      }
      work_sync();
      const uint16_t* stage_c = stage;
      for (int x = tid - kWorkWarp0 * 32; x < kM * (kD / 8); x += kWorkWarps * 32) {
        const int h = x / (kD / 8), c8 = x % (kD / 8);
        const uint32_t dst = (uint32_t)(h / hp);
        const int slot = (int)rank * hp + (h - (int)dst * hp);
        dsmem_st_u32x4(dsmem_map(&pin[slot * kD + c8 * 8], dst),
                       *reinterpret_cast<const uint4*>(&stage_c[h * kD + c8 * 8]));
      }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // (D) every run's partials of this CTA's heads are here
    // heads [rank * hp, (rank + 1) * hp): combine the runs' partials (a run without keys has
    // maximum -inf and weight 0)
    const int hb0 = (int)rank * hp, hb1 = min(kM, hb0 + hp);
    constexpr int C4 = kD / 4;
    for (int x = tid; x < (hb1 - hb0) * C4; x += kThreads) {
      const int hl = x / C4, c4 = x % C4;
      const int h = hb0 + hl;
      if (h >= p.H) continue;
      float Mx = -INFINITY;
      for (uint32_t sp = 0; sp < C; ++sp) Mx = fmaxf(Mx, pinml[sp * hp + hl].x);
      float Lx = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      if (Mx != -INFINITY) {
        for (uint32_t sp = 0; sp < C; ++sp) {
          const float2 ml = pinml[sp * hp + hl];
          if (ml.x == -INFINITY || ml.y <= 0.f) continue;
          const float wl = exp2f((ml.x - Mx) * kLog2e) * ml.y;  // the run's weight: e^(m - M) l
          const uint2 pv = *reinterpret_cast<const uint2*>(&pin[(sp * hp + hl) * kD + c4 * 4]);
          Lx += wl;
          acc.x += wl * bf16_bits_to_f32(pv.x & 0xFFFFu);
          acc.y += wl * bf16_bits_to_f32(pv.x >> 16);
          acc.z += wl * bf16_bits_to_f32(pv.y & 0xFFFFu);
          acc.w += wl * bf16_bits_to_f32(pv.y >> 16);
        }
      }
      const float inv = Lx > 0.f ? 1.f / Lx : 0.f;
      uint2 pk2;
      pk2.x = pack_bf16x2(acc.x * inv, acc.y * inv);
      pk2.y = pack_bf16x2(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(p.out + (b * p.H + h) * kD + c4 * 4) = pk2;
      if (p.lse != nullptr && c4 == 0) p.lse[b * p.H + h] = Lx > 0.f ? Mx + logf(Lx) : -INFINITY;
    }
  }
  pdl_wait();  // completion stays ordered after the predecessor's (no-op if already waited)
  // Without the attention the last remote stores (the selection's counts) precede barrier (B),
  // and with it the last ones precede (D): no CTA touches another's shared memory after that,
  // so the CTAs leave without a further cluster barrier.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int g_max_active[kMaxDevicesDecode][kDecodeMaxCluster + 1];

}  // namespace

// Plans the fused step: the cluster size C (each sequence's entries split over C CTAs) that
// minimises the estimated time over the waves of co-resident clusters, within the kernel's
// limits (at most kDecodeFusedChunk entries per CTA, kDecodeMaxKeys attention keys per CTA).
DecodePlan plan_decode(int B, int64_t E, int64_t n_vis, int k, int W, bool attend,
                       bool want_scores) {
  DecodePlan best{};
  best.ok = false;
  const bool select_all = n_vis <= k;
  const bool scoring = !select_all || want_scores;
  // key copies move whole 16-byte runs of scales: E % 8 == 0 (nothing is copied when every
  // visible entry is selected and no score is requested)
  if (B < 1 || n_vis < 0 || k < 1 || k > kDecodeMaxSel || (scoring && E % 8 != 0)) return best;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesDecode) return best;
  const int64_t tiles = (n_vis + kTileM - 1) / kTileM;
  const int64_t cnt = n_vis < k ? n_vis : k;
  const int64_t nw = W;  // the window is at most W tokens
  double best_t = 1e30;
  for (int C = kDecodeMaxCluster; C >= 1; --C) {
    const int64_t chunk = (tiles + C - 1) / C * kTileM;
    // Longer chunks stream more key bytes through one SM than the separate indexer spreads
    // over the whole GPU: measured slower there, with and without the attention (4 rows of
    // 262144 entries in 16-CTA clusters: 39 us for scores and selection against 27 + 17 us for
    // the separate indexer and top-k, whose step overlaps better with a concurrent layer).
    if (chunk > kDecodeFusedChunk) continue;
    const int64_t P = (cnt + nw + C - 1) / C;
    if (attend && P > kDecodeMaxKeys) continue;
    int act = g_max_active[dev][C];
    if (act == 0) {
      auto kern = csa_decode_kernel;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBytes) != cudaSuccess ||
          cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
              cudaSuccess)
        return best;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)C, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)C;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&act, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        act = 0;
      }
      g_max_active[dev][C] = act > 0 ? act : -1;
    }
    if (act <= 0) continue;
    const int64_t waves = (B + act - 1) / act;
    // per-CTA estimate in microseconds: its key bytes at ~47 GB/s per SM, its attention rows,
    // and a fixed cost for the launch, the cluster rounds and the merge
    const double t = (double)waves * ((double)chunk * 34.0 / 47e3 +
                                      (attend ? (double)P * 512.0 / 47e3 : 0.0) + 3.0);
    if (t < best_t - 1e-9) {
      best_t = t;
      best.ok = true;
      best.C = C;
      best.chunk = (int)chunk;
      best.P = (int)(attend ? P : 0);
    }
  }
  return best;
}

namespace {
DecParams decode_params(const DecodeArgs& a, const DecodePlan& pl, uint32_t* status) {
  DecParams p;
  p.qi_codes = a.qi_codes;
  p.qi_scales = a.qi_scales;
  p.ki_codes = a.ki_codes;
  p.ki_scales = a.ki_scales;
  p.scores = a.scores;
  p.topk_idx = a.topk_idx;
  p.topk_cnt = a.topk_cnt;
  p.E = a.E;
  p.t = a.t;
  p.m = a.m;
  p.k = a.k;
  p.H_I = a.H_I;
  const int64_t nv = std::min<int64_t>(a.E, (a.t + 1) / a.m);
  p.n_vis = (int)(nv < 0 ? 0 : nv);
  p.chunk = pl.chunk;
  p.keys_fresh_from = a.keys_fresh_from;
  p.wait_first = a.wait_first ? 1 : 0;
  p.attend = a.attend ? 1 : 0;
  p.H = a.H;
  p.W = a.W;
  p.P = pl.P;
  p.q = a.q;
  p.k_cmp = a.k_cmp;
  p.v_cmp = a.v_cmp;
  p.k_raw = a.k_raw;
  p.v_raw = a.v_raw;
  p.out = a.out;
  p.lse = a.lse;
  p.N = a.N;
  p.logits = a.logits;
  p.pool_j0 = a.pool_j0;
  p.pool_j1 = a.pool_j1;
  p.status = status;
  const FaultConfig fc = fault_config();
  p.wait_budget = fc.wait_budget;
  p.fault_mask = fc.skip_mask;
  p.split = 0;
  return p;
}
}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& pl, uint32_t* status,
                          cudaStream_t stream) {
  if (!pl.ok) return cudaErrorInvalidValue;
  const DecParams p = decode_params(a, pl, status);
  auto kern = csa_decode_kernel;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  if (pl.C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  ProfScope prof(stream, a.attend ? "csa_decode" : "indexer_topk");
  return launch_ex(kern, dim3((unsigned)(a.B * pl.C)), dim3(kThreads), kSmemBytes, stream,
                   (unsigned)pl.C, p);
}

// Scores only: every sequence's visible entries split evenly over `split` CTAs (one wave of one
// CTA per SM where the batch allows), each at most kDecodeMaxChunk entries.
bool plan_decode_scores(int B, int64_t E, int64_t n_vis, int* split, int* chunk) {
  if (B < 1 || n_vis < 1 || E % 8 != 0) return false;
  const int64_t tiles = (n_vis + kTileM - 1) / kTileM;
  int64_t sp = std::max<int64_t>(1, kNumSMs / B);
  sp = std::min<int64_t>(sp, tiles);
  const int64_t ch = (tiles + sp - 1) / sp * kTileM;
  if (ch > kDecodeMaxChunk) return false;
  *split = (int)sp;
  *chunk = (int)ch;
  return true;
}

cudaError_t launch_decode_scores(const DecodeArgs& a, int split, int chunk, uint32_t* status,
                                 cudaStream_t stream) {
  if (split < 1 || chunk < 1 || chunk > kDecodeMaxChunk || a.scores == nullptr)
    return cudaErrorInvalidValue;
  DecodePlan pl{};
  pl.ok = true;
  pl.C = 1;
  pl.chunk = chunk;
  pl.P = 0;
  DecodeArgs b = a;
  b.attend = false;
  if (b.pool_j1 < b.pool_j0) b.pool_j1 = b.pool_j0;  // none
  DecParams p = decode_params(b, pl, status);
  p.split = split;
  auto kern = csa_decode_kernel;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  ProfScope prof(stream, "indexer_mxf4");
  return launch_ex(kern, dim3((unsigned)(a.B * split)), dim3(kThreads), kSmemBytes, stream, 1u,
                   p);
}

}  // namespace csa
