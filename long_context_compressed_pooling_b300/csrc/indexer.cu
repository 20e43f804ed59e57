// Lightning Indexer scores on the 5th-generation tensor cores (tcgen05, FP4).
//
// 9fzt.com DeepSeek-V4 summary, item 4: the CSA indexer's QK path runs in FP4 and its scores
// are reduced from FP32 to BF16 before the top-k selector. Lighthouse "deep deepseek v4
// release" 八.7: the indexer keeps its own compressed keys.
//   s[b,i,j] = bf16_rne( sum_h max(0, q_I[b,i,h] . k_I[b,j]) )
// with q_I, k_I block-scaled FP4 vectors (e2m1 codes, one UE8M0 scale per 32 elements).
//
// Layout of the contraction. A = the entries' FP4 index keys (M = 128 entries per tile,
// K = 64 e2m1 values = 32 bytes per row).
// Decode (one query per sequence): B = one row per (query, head, 32-element block) holding that
// block's codes and zeros elsewhere, so D[j, (q,h,blk)] is the UNSCALED partial dot product of
// one scale block, every scale factor is 1.0 and the UE8M0 scales are applied in the epilogue as
// exact power-of-two multiplies. With d_I = 64 a tile is 4 KB contiguous in HBM and arrives with
// ONE bulk copy (a tensor-map box with 32-byte rows would cost 128 small TMA requests per tile);
// it lands unswizzled while the MMA reads it through the 32-byte swizzle, which swaps the two
// 16-byte halves of rows whose bit 2 is set. Those rows therefore meet the query blocks in
// swapped positions, so B carries each head twice (blocks in place, blocks swapped) and every
// epilogue thread reads the pair that matches its row.
// Prefill (a query group per CTA, swizzled TMA tiles): B = one row per (query, head) with both
// blocks, and the block scales of entries (A) and queries (B) are the MMA's scale factors, so
// D[j, (q,h)] is the head's scaled dot product and the epilogue only takes ReLU, sums the heads
// and rounds. The A scale factors change with every tile: one region per accumulator group,
// rewritten by the epilogue before it releases the group to the next tile (row i of a tile: lane
// i, column i / 32; byte k of the word scales block k). d_I = 32 rows (16 B) are zero-padded to
// 32 bytes (the TMA box is zero-filled, B's second block is zero).
// Exactness: a block's partial sum of e2m1 products is a multiple of 1/4 below 2^11, a scaled
// block sum a multiple of 2^-10 below 2^12 for the workloads' scales (2^-4..2^0), so the fp32
// sums, in the tensor core or in the epilogue, are exact (a GPU probe confirmed it for the
// scaled two-block accumulation) and the BF16 rounding is the only rounding, as the method
// specifies.
//
// Pipeline. A copy warp fills a 3-slot ring (8 tiles per slot: one bulk copy of codes and one
// of scales per slot, since each copy instruction costs ~0.3 us to issue whatever its size); it
// starts at once and never joins the set-up barriers of the other warps. A slot is refilled only
// after the MMAs that read its codes have completed AND every epilogue warp has finished the
// slot's last group (the epilogue reads the slot's scale tile). The MMA warp issues
// groups of G tiles (one elected lane of a converged warp) into the next accumulator group of a
// ring in tensor memory (3 x 4 x 16 columns for decode, 2 x 1 x 224 for prefill) and commits
// once per group; the epilogue warps (two per tensor-memory lane quarter for decode, four for
// prefill) drain a group
// together, so the commit -> epilogue round trip is paid once per group. Decode (one query per
// sequence) runs persistent CTAs over all (sequence, tile) pairs; prefill gives each CTA one
// (sequence, query group). Every mbarrier wait is bounded (kFlagTimeout on expiry).
#include "common.cuh"
#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

constexpr int kTileM = 128;
constexpr int kRowBytes = 32;
constexpr int kATileBytes = kTileM * kRowBytes;
constexpr int kSlotTiles = 8;   // tiles per copy slot (one code copy + one scale copy)
constexpr int kSlots = 3;       // slots in the ring
constexpr int kRingTiles = kSlotTiles * kSlots;
constexpr int kScaleTileBytes = kTileM * 2;  // one tile's UE8M0 scales (NB = 2)
// Copy warp, MMA warp and EW epilogue warps per tensor-memory lane quarter (2 for decode, whose
// CTAs run two per SM; 4 for prefill, whose epilogue is the critical path).
constexpr int threads_for(int ew) { return 64 + 128 * ew; }
constexpr int kMaxCols = 224;    // MMA N of a prefill CTA (14 queries x 16 columns)
constexpr int kMaxG = 4;
constexpr int kMaxAcc = 8;  // accumulator groups in tensor memory (a ring)
// Scale-factor regions in tensor memory (kind::mxf4 scale_vec::2X), each starting on a 16-column
// boundary. A: row i in lane i, column i / 32 (all 1.0: the entries' scales are applied in the
// epilogue). B: column n of the MMA in lane 32 q + n % 32 of every lane quarter q, column n / 32.
constexpr int kSfCols = 16;
constexpr int kMaxSeqPerCta = 8;  // decode: query operands of up to 8 sequences stay resident

struct IdxParams {
  const uint8_t* qi_codes;   // [B, Nq, H_I, NB*16]
  const uint8_t* qi_scales;  // [B, Nq, H_I, NB]
  const uint8_t* ki_scales;  // [B, E, NB]
  uint16_t* scores;          // [B, Nq, E]
  float* scores_f32;         // optional [B, Nq, E]: the exact FP32 scores before BF16 rounding
  int64_t q_pos0, E;
  int Nq, m, QN, ncols, G, nacc, n_splits, tmem_cols;
  int B, tiles_per_seq;      // decode: CTAs walk contiguous ranges of (sequence, tile)
  int64_t total_tiles;
  const uint8_t* ki_codes;   // [B, E, 32] (bulk-copy path)
  uint32_t* status;
  // paged cache (bulk-copy path only): the keys of entry j of sequence b are row
  // (page << page_shift) + (j & page_mask) of the key pools, page = block_table[b][j >> page_shift]
  const int32_t* block_table;
  int max_blocks, n_pages, page_shift;
  // Inputs a predecessor kernel on the stream may still be writing (it lets this kernel start
  // early): key tiles holding an entry at or above keys_fresh_from are copied only after the
  // grid-dependency wait, and with q_fresh set the query operands are read only after it.
  int64_t keys_fresh_from;
  int q_fresh;
  long long wait_budget;  // bounded-wait budget (SM cycles)
  uint32_t fault_mask;    // kFault* switches set by a failure-injection test (0 otherwise)
};

// Shared memory for a launch whose B operand has `brows` rows (decode: 8 sequences x ncols;
// prefill: ncols), so that decode CTAs stay small enough for two per SM.
constexpr size_t smem_bytes(int brows) {
  return 1024 /*align slack*/ + kRingTiles * kATileBytes + kRingTiles * kScaleTileBytes +
         (size_t)brows * kRowBytes + (size_t)brows * sizeof(float) + kMaxCols * sizeof(int64_t) +
         (2 * kSlots + 2 * kMaxAcc + 3) * 8 + 64;
}

// Named barrier over every warp but the copy warp (the copy warp never waits on set-up).
CSA_DEV void work_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// H_I heads, NB = d_I / 32 scale blocks per vector, SW = 2 for the bulk-copy path (each head's
// blocks in place and swapped), else 1; CPQ = H_I * NB * SW MMA columns per query.
// F32OUT: also write the exact FP32 scores (p.scores_f32); a separate instantiation so that the
// path without them carries no extra instruction in its issue-bound epilogue.
template <int H_I, int NB, int SW, bool PREFILL, bool F32OUT, int EW = PREFILL ? 4 : 2>
__global__ void __launch_bounds__(threads_for(EW)) indexer_kernel(const __grid_constant__ CUtensorMap kmap,
                                                           const IdxParams p) {
  // Prefill puts both blocks' UE8M0 scales of entries (A) and queries (B) into the MMA, which
  // then accumulates the two scaled block sums of a head into one column (exact, like every
  // partial sum here); decode keeps one column per block and applies the scales afterwards.
  constexpr int CPQ = PREFILL ? H_I : H_I * NB * SW;
  static_assert(16 % CPQ == 0, "columns per query must divide 16");
  static_assert(!PREFILL || SW == 1, "prefill reads its key tiles through the tensor map");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* atiles = base;                                    // kRingTiles x 4096, 1024-aligned
  const int brows = (p.Nq == 1 ? kMaxSeqPerCta : 1) * p.ncols;
  uint8_t* btile = atiles + kRingTiles * kATileBytes;        // brows x 32, 1024-aligned
  uint8_t* stiles = btile + brows * kRowBytes;               // bulk path: kRingTiles x 256 B
  uint32_t* qbyte = reinterpret_cast<uint32_t*>(stiles + kRingTiles * kScaleTileBytes);
  int64_t* qvis = reinterpret_cast<int64_t*>(qbyte + brows);  // visible entries per query
  uint64_t* bars = reinterpret_cast<uint64_t*>(qvis + kMaxCols);
  uint64_t* full = bars;                 // [kSlots]
  uint64_t* empty = bars + kSlots;       // [kSlots]
  uint64_t* tfull = bars + 2 * kSlots;   // [kMaxAcc]
  uint64_t* tempty = tfull + kMaxAcc;    // [kMaxAcc]
  uint64_t* drain = tempty + kMaxAcc;    // [1]
  uint64_t* done = drain + 1;            // [1] every epilogue warp finished with TMEM
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  int* aborted = reinterpret_cast<int*>(tmem_slot + 1);

  pdl_trigger();
  // Work: prefill (Nq > 1) -> one (sequence, query group) per grid (y, z) and a range of entry
  // tiles per x. Decode (Nq == 1) -> CTA x walks the flattened (sequence, tile) range
  // [tb, te) of all sequences; the query operands of the sequences it touches stay resident.
  constexpr bool decode = !PREFILL;  // the launch picks PREFILL = (Nq > 1)
  // The entries' UE8M0 scales (two per entry) travel with their codes into the slot ring (bulk
  // copies need 16-byte aligned runs: E % 8 == 0, always true on the bulk-copy path); otherwise
  // the epilogue reads them from global memory.
  const bool scales_in_smem = SW == 2 || (NB == 2 && (p.E % 8) == 0);
  const int split = blockIdx.x, group = blockIdx.y;
  const int i0 = decode ? 0 : group * p.QN;
  const int nq = decode ? 1 : min(p.QN, p.Nq - i0);
  int64_t tb, te;
  int b_first;
  if (decode) {
    // total * split / n in 32-bit arithmetic (64-bit division is emulated): total = a n + r,
    // so total * split / n = a split + r split / n with r split < n^2 (the launch keeps
    // total_tiles < 2^31 and n_splits < 2^15)
    const uint32_t T = (uint32_t)p.total_tiles, n = (uint32_t)p.n_splits;
    const uint32_t a = T / n, r = T % n, sp = (uint32_t)split;
    tb = (int64_t)(a * sp + r * sp / n);
    te = (int64_t)(a * (sp + 1) + r * (sp + 1) / n);
    b_first = (int)((uint32_t)tb / (uint32_t)p.tiles_per_seq);
  } else {
    const int64_t t_last = p.q_pos0 + i0 + nq - 1;
    const int64_t nv_max = min(p.E, (t_last + 1) / p.m);
    const int64_t tiles = (nv_max + kTileM - 1) / kTileM;
    tb = tiles * split / p.n_splits;
    te = tiles * (split + 1) / p.n_splits;
    b_first = blockIdx.z;
  }
  if (tb >= te) return;  // uniform over the CTA
  const int ntiles = (int)(te - tb);
  const int n_seq =
      decode ? (int)((uint32_t)(te - 1) / (uint32_t)p.tiles_per_seq) - b_first + 1 : 1;
  if (n_seq > kMaxSeqPerCta) {  // the launch plan never produces this; refuse rather than overflow
    if (threadIdx.x == 0) atomicOr(p.status, kFlagBadIndex);
    return;
  }
  const int G = p.G;                      // tiles per MMA / epilogue group (divides kSlotTiles)
  const int ngroups = (ntiles + G - 1) / G;
  const int nunits = (ntiles + kSlotTiles - 1) / kSlotTiles;  // copy slots to fill
  // Tile `it` of this CTA -> (sequence, first entry) with 32-bit arithmetic only (64-bit
  // integer division is emulated in software and must stay out of the loops).
  const int tps = p.tiles_per_seq;
  const int t_first = decode ? (int)(tb - (int64_t)b_first * tps) : (int)tb;
  auto tile_seq = [&](int it) -> int {
    return decode ? b_first + (int)((unsigned)(t_first + it) / (unsigned)tps) : b_first;
  };
  auto tile_row0 = [&](int it) -> int {
    const unsigned t = (unsigned)(t_first + it);
    return (int)(decode ? t % (unsigned)tps : t) * kTileM;
  };
  auto ring_tile = [&](int it) -> int {  // position of tile `it` in the shared-memory ring
    return ((it / kSlotTiles) % kSlots) * kSlotTiles + it % kSlotTiles;
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWork = threads_for(EW) - 32;  // every warp but the copy warp
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1 + 4 * EW);  // the MMAs' commit + every epilogue warp
    }
    for (int a = 0; a < p.nacc; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4 * EW);
    }
    mbar_init(drain, 1);
    mbar_init(done, 4 * EW);
    *aborted = 0;
    fence_mbar_init();
    prefetch_tensormap(&kmap);
  }
  __syncwarp();
  __syncthreads();

  if (warp == 0) {
    // ---------------- copy warp: fills the ring slot by slot, never joins the set-up ----------
    // Key tiles below keys_fresh_from cannot be written by the kernel this one overlaps, so they
    // are copied at once; the first slot holding a tile at or above it is issued only after the
    // grid-dependency wait (the predecessor, e.g. the pooling of the step's new index keys, has
    // then completed and its writes are visible). Every bulk copy costs ~0.3 us to issue
    // whatever its size, so a slot (8 tiles) is one code copy and one scale copy whenever the
    // tiles form one contiguous span of HBM (always, unless a ragged sequence tail intervenes).
    // A page holds whole tiles, so a paged tile is always copied whole (its rows past the
    // visible entries are never scored).
    auto tile_bytes = [&](int it) -> uint32_t {  // rows that exist in this tile x 32 B
      if (p.block_table) return (uint32_t)kTileM * kRowBytes;
      return (uint32_t)min((int64_t)kTileM, p.E - (int64_t)tile_row0(it)) * kRowBytes;
    };
    auto tile_addr = [&](int it) -> int64_t {  // entry (pool row) of the tile's first row
      if (p.block_table) {
        const int j = tile_row0(it);
        const int blk = j >> p.page_shift;
        int pg = blk < p.max_blocks ? p.block_table[(int64_t)tile_seq(it) * p.max_blocks + blk] : -1;
        if (pg < 0 || pg >= p.n_pages) {
          atomicOr(p.status, kFlagBadIndex);  // unmapped page: scores of page 0, flagged
          pg = 0;
        }
        return ((int64_t)pg << p.page_shift) + (j & ((1 << p.page_shift) - 1));
      }
      return (int64_t)tile_seq(it) * p.E + tile_row0(it);
    };
    auto issue_unit = [&](int u) {
      const int slot = u % kSlots;
      const int t0 = u * kSlotTiles, t1 = min(ntiles, t0 + kSlotTiles);
      if (SW == 2) {
        uint32_t bytes = 0;
        for (int it = t0; it < t1; ++it) bytes += tile_bytes(it) + tile_bytes(it) / 16;
        mbar_arrive_expect_tx(&full[slot], bytes);
        int a = t0;
        while (a < t1) {
          const int64_t e0 = tile_addr(a);
          uint32_t rows = tile_bytes(a) / kRowBytes;
          int b = a + 1;
          while (b < t1 && rows == (uint32_t)(b - a) * kTileM && tile_addr(b) == e0 + rows) {
            rows += tile_bytes(b) / kRowBytes;
            ++b;
          }
          const int rt = ring_tile(a);
          bulk_load(atiles + rt * kATileBytes, p.ki_codes + e0 * kRowBytes, rows * kRowBytes,
                    &full[slot]);
          bulk_load(stiles + rt * kScaleTileBytes, p.ki_scales + e0 * 2, rows * 2, &full[slot]);
          a = b;
        }
      } else {
        uint32_t bytes = (uint32_t)((t1 - t0) * kATileBytes);
        if (scales_in_smem)
          for (int it = t0; it < t1; ++it) bytes += tile_bytes(it) / 16;
        mbar_arrive_expect_tx(&full[slot], bytes);
        for (int it = t0; it < t1; ++it)
          tma_load_3d(atiles + ring_tile(it) * kATileBytes, &kmap, &full[slot], 0, tile_row0(it),
                      tile_seq(it));
        if (scales_in_smem) {  // the tiles' scale bytes, one copy per contiguous run
          int a = t0;
          while (a < t1) {
            const int64_t e0 = tile_addr(a);
            uint32_t rows = tile_bytes(a) / kRowBytes;
            int b = a + 1;
            while (b < t1 && rows == (uint32_t)(b - a) * kTileM && tile_addr(b) == e0 + rows) {
              rows += tile_bytes(b) / kRowBytes;
              ++b;
            }
            bulk_load(stiles + ring_tile(a) * kScaleTileBytes, p.ki_scales + e0 * 2, rows * 2,
                      &full[slot]);
            a = b;
          }
        }
      }
    };
    // first slot that holds a tile the predecessor may still be writing (nunits: none)
    int fresh_unit = nunits;
    for (int it = 0; it < ntiles; ++it)
      if ((int64_t)tile_row0(it) + kTileM > p.keys_fresh_from) {
        fresh_unit = it / kSlotTiles;
        break;
      }
    bool waited = false;
    // the first kSlots units go to free slots: one lane each, issued together
    const int first = min(kSlots, nunits);
    if (fresh_unit < first) {
      pdl_wait();
      waited = true;
    }
    if (p.fault_mask & kFaultSkipKeyCopies) {  // failure injection: no tile ever arrives
      if (!waited) pdl_wait();
      return;
    }
    if (lane < first) issue_unit(lane);
    __syncwarp();
    int issued = first;
    for (int u = first; u < nunits; ++u) {
      const int slot = u % kSlots, use = u / kSlots;
      if (!mbar_wait_warp(&empty[slot], (uint32_t)(use - 1) & 1u, p.status, p.wait_budget)) {
        if (lane == 0) *aborted = 1;
        break;
      }
      if (!waited && u >= fresh_unit) {
        pdl_wait();
        waited = true;
      }
      if (elect_one()) issue_unit(u);
      __syncwarp();
      issued = u + 1;
    }
    // stay until this CTA's own copies have landed (the MMA warp normally sees them first)
    for (int u = max(0, issued - kSlots); u < issued; ++u)
      mbar_wait_warp(&full[u % kSlots], (uint32_t)(u / kSlots) & 1u, p.status, p.wait_budget);
    return;
  }

  // ---- set-up of the work warps: B operand, query scales, visibility, TMEM, scale factors ----
  // Sequence sl of this CTA owns B rows [sl * ncols, (sl + 1) * ncols).
  if (p.q_fresh) pdl_wait();  // the queries may be the predecessor's output
  const int wt = threadIdx.x - 32;
  for (int idx = wt; idx < n_seq * p.ncols * 2; idx += kWork) {
    const int rr = idx >> 1, c = idx & 1;
    const int sl = rr / p.ncols, r = rr % p.ncols;
    const int ql = r / CPQ, h = PREFILL ? r % H_I : (r / (NB * SW)) % H_I,
              sw = (r / NB) % SW, blk = PREFILL ? c : r % NB;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    // prefill: row (query, head) holds both blocks; decode: one block per row, zeros elsewhere
    if (ql < nq && (PREFILL ? c < NB : c == (blk ^ sw))) {
      const uint8_t* src = p.qi_codes +
          (((int64_t)(b_first + sl) * p.Nq + i0 + ql) * H_I + h) * (NB * 16) + blk * 16;
      v = *reinterpret_cast<const uint4*>(src);
    }
    const int phys = rr * kRowBytes + ((c ^ ((rr >> 2) & 1)) << 4);  // 32-byte swizzle
    *reinterpret_cast<uint4*>(btile + phys) = v;
  }
  for (int rr = wt; rr < n_seq * p.ncols; rr += kWork) {
    const int sl = rr / p.ncols, r = rr % p.ncols;
    const int ql = r / CPQ;
    const int64_t qrow = ((int64_t)(b_first + sl) * p.Nq + i0 + ql) * H_I;
    if constexpr (PREFILL) {
      // the row's scale-factor word: byte 0 scales block 0, byte 1 block 1 (1.0 elsewhere)
      const int h = r % H_I;
      uint32_t w = 0x7F7F7F7Fu;
      if (ql < nq) {
        w = 0x7F7F0000u | p.qi_scales[(qrow + h) * NB];
        w |= (NB == 2 ? (uint32_t)p.qi_scales[(qrow + h) * NB + 1] : 127u) << 8;
      }
      qbyte[rr] = w;
    } else {
      const int h = (r / (NB * SW)) % H_I, blk = r % NB;
      qbyte[rr] = ql < nq ? (uint32_t)p.qi_scales[(qrow + h) * NB + blk]
                          : 127u;  // scale 1.0 for the zero rows of absent queries
    }
  }
  for (int ql = wt; ql < nq; ql += kWork)
    qvis[ql] = min(p.E, (p.q_pos0 + i0 + ql + 1) / p.m);
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  __syncwarp();
  tc_fence_before();
  work_sync(kWork);
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t acc_cols = (uint32_t)(G * p.ncols);  // one accumulator group
  // scale-factor regions, each on a 16-column boundary: A (prefill: one per accumulator group,
  // rewritten for every tile), then B
  const uint32_t sfa_col = (uint32_t)p.nacc * acc_cols;
  const uint32_t sfb_col = sfa_col + (uint32_t)(PREFILL ? p.nacc : 1) * kSfCols;
  // Prefill (one sequence per CTA): every B column carries its query block's UE8M0 scale, so the
  // MMA yields scale x (exact partial sum of e2m1 products), still exact. Decode CTAs may hold
  // several sequences behind one scale region: their B scales stay 1.0 and the query scales are
  // applied in the epilogue.
  constexpr bool q_in_mma = PREFILL;
  if (warp >= 2 && warp < 6) {
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    for (uint32_t c = sfa_col; c < sfb_col + kSfCols; c += 8)
      tmem_st8_fill(tmem + lane_base + c, 0x7F7F7F7Fu);
    if (q_in_mma) {
      tmem_st_wait();
      for (int c = 0; c < (p.ncols + 31) / 32; ++c) {
        const int n = c * 32 + lane;
        const uint32_t w = n < p.ncols ? qbyte[n] : 0x7F7F7F7Fu;
        tmem_st1(tmem + lane_base + sfb_col + (uint32_t)c, PREFILL ? w : w * 0x01010101u);
      }
    }
    tmem_st_wait();
  }
  __syncwarp();
  tc_fence_before();
  work_sync(kWork);
  tc_fence_after();
  pdl_wait();  // the predecessor may still read the score buffer this kernel writes

  if (warp == 1) {
    // ---------------- MMA issuer (whole warp, one elected lane issues) ----------------
    const uint32_t idesc = idesc_mxf4(kTileM, p.ncols);
    for (int g = 0; g < ngroups; ++g) {
      const int u = g * G / kSlotTiles;
      const int slot = u % kSlots;
      const int a = g % p.nacc;
      const uint32_t aph = (uint32_t)(g / p.nacc) & 1u;
      // (prefill: the epilogue's first round of arrivals says the buffer's tile scales are in)
      if (!mbar_wait_warp(&tempty[a], PREFILL ? aph : aph ^ 1u, p.status, p.wait_budget) ||
          !mbar_wait_warp(&full[slot], (uint32_t)(u / kSlots) & 1u, p.status, p.wait_budget)) {
        if (lane == 0) *aborted = 1;
        break;
      }
      tc_fence_after();
      const int nt = min(G, ntiles - g * G);
      const bool unit_done = (g + 1) * G >= min(ntiles, (u + 1) * kSlotTiles);
      if (elect_one()) {
        for (int i = 0; i < nt; ++i) {
          const int it = g * G + i;
          const uint64_t adesc =
              smem_desc(smem_addr(atiles + ring_tile(it) * kATileBytes), 16, 256, kSwizzle32B);
          const uint64_t bdesc = smem_desc(
              smem_addr(btile + (tile_seq(it) - b_first) * p.ncols * kRowBytes), 16, 256,
              kSwizzle32B);
          umma_mxf4(tmem + (uint32_t)(a * acc_cols + i * p.ncols), adesc, bdesc, idesc,
                    tmem + sfa_col + (PREFILL ? (uint32_t)a * kSfCols : 0u), tmem + sfb_col, 0u);
        }
        if (unit_done) umma_commit(&empty[slot]);  // the slot's last group frees the slot
        umma_commit(&tfull[a]);
      }
      __syncwarp();
    }
    if (elect_one()) umma_commit(drain);  // arrives once every MMA above has finished
    __syncwarp();
    mbar_wait_warp(drain, 0, p.status, p.wait_budget);
  } else {
    // ---------------- epilogue: 8 warps, two per tensor-memory lane quarter ----------------
    const int quarter = warp & 3;
    const int sub = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const bool swapped = SW == 2 && ((row >> 2) & 1);  // unswizzled row read through the swizzle
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int cchunks = p.ncols / 16;
    // Prefill: warp 0 of each lane quarter writes the entry scales of tile `it` into the A
    // scale region of accumulator group `a` (row i of the tile: lane i, column i / 32, byte k
    // scaling block k), once the tile's scales are in shared memory (or from global memory).
    auto write_sfa = [&](int it, int a) -> bool {
      if (scales_in_smem) {
        const int u = it / kSlotTiles;
        if (!mbar_wait_warp(&full[u % kSlots], (uint32_t)(u / kSlots) & 1u, p.status,
                            p.wait_budget))
          return false;
      }
      const int64_t j = (int64_t)tile_row0(it) + row;
      uint32_t sb = 0x7F7Fu;
      if (j < p.E) {
        if (scales_in_smem)
          sb = *reinterpret_cast<const uint16_t*>(stiles + ring_tile(it) * kScaleTileBytes +
                                                  row * 2);
        else
          sb = NB == 2 ? (uint32_t)*reinterpret_cast<const uint16_t*>(
                             p.ki_scales + ((int64_t)b_first * p.E + j) * 2)
                       : (uint32_t)p.ki_scales[(int64_t)b_first * p.E + j];
        if (NB == 1) sb = (sb & 0xFFu) | 0x7F00u;
      }
      tmem_st1(tmem + lane_base + sfa_col + (uint32_t)(a * kSfCols + quarter), 0x7F7F0000u | sb);
      tmem_st_wait();
      return true;
    };
    if constexpr (PREFILL) {
      // the first tile of every accumulator group; this round of arrivals tells the MMA warp
      bool ok = true;
      if (sub == 0)
        for (int a = 0; a < p.nacc && a < ntiles && ok; ++a) ok = write_sfa(a, a);
      if (!ok && lane == 0) *aborted = 1;
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        for (int a = 0; a < p.nacc; ++a) mbar_arrive(&tempty[a]);
    }
    for (int g = 0; g < ngroups; ++g) {
      const int a = g % p.nacc;
      const uint32_t aph = (uint32_t)(g / p.nacc) & 1u;
      const int unit = g * G / kSlotTiles;
      const int slot = unit % kSlots;
      // The slot's scale tile is read below: acquire the copy that filled it (its phase is
      // complete, and it cannot be refilled before this warp releases it).
      if (!mbar_wait_warp(&tfull[a], aph, p.status, p.wait_budget) ||
          (scales_in_smem && !mbar_wait_warp(&full[slot], (uint32_t)(unit / kSlots) & 1u,
                                             p.status, p.wait_budget))) {
        if (lane == 0) *aborted = 1;
        break;
      }
      tc_fence_after();
      const int nt = min(G, ntiles - g * G);
      const bool unit_done = (g + 1) * G >= min(ntiles, (unit + 1) * kSlotTiles);
      if constexpr (PREFILL) {
        // One tile per group (G = 1); warp `sub` of the quarter owns the 16-column chunks
        // sub, sub + EW, ..., read two per tensor-memory round trip.
        constexpr int kChunksPerWarp = (kMaxCols / 16 + EW - 1) / EW;
        const int it = g;
        const int64_t j = (int64_t)tile_row0(it) + row;
        uint16_t* srow = p.scores + ((int64_t)b_first * p.Nq + i0) * p.E + j;
        // every query of the group sees the whole tile (the common case away from the causal
        // edge): no per-score visibility test
        const bool all_vis = (int64_t)tile_row0(it) + kTileM <= (int64_t)qvis[0];
#pragma unroll
        for (int k0 = 0; k0 < kChunksPerWarp; k0 += 2) {
          uint32_t r[2][16];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c = sub + (k0 + k) * EW;
            if (c < cchunks)
              tmem_ld16(tmem + lane_base + (uint32_t)(a * acc_cols + c * 16), r[k]);
          }
          tmem_ld_wait();
          if (j >= p.E) continue;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c = sub + (k0 + k) * EW;
            if (c < cchunks) {
#pragma unroll
              for (int cc = 0; cc < 16; cc += CPQ) {
                const int ql = (c * 16 + cc) / CPQ;
                if (ql < nq) {
                  // column (query, head) holds the head's exact scaled dot product; the ReLU
                  // acts on the bit patterns (negative values and -0 become +0), so the sum of
                  // the non-negative terms is never -0 (the terms are exact: any order)
                  float sc = __int_as_float(max((int)r[k][cc], 0));
#pragma unroll
                  for (int h = 1; h < H_I; ++h) sc += __int_as_float(max((int)r[k][cc + h], 0));
                  if (all_vis || j < qvis[ql]) {
                    srow[(int64_t)ql * p.E] = f32_to_bf16_bits(sc);
                    if constexpr (F32OUT)
                      p.scores_f32[(srow - p.scores) + (int64_t)ql * p.E] = sc;
                  }
                }
              }
            }
          }
        }
      } else {
        // units (tile i, 16-column chunk) of the group, split over the quarter's EW warps; two
        // units per tensor-memory round trip
        // (prefill groups hold one tile; decode tiles have one or two chunks: no divisions)
        const int nunits_g = nt * cchunks;
        const int csh = cchunks == 2 ? 1 : 0;
        for (int u0 = sub; u0 < nunits_g; u0 += 2 * EW) {
          const int uu[2] = {u0, u0 + EW};
          int ui[2], uc[2];
  #pragma unroll
          for (int x = 0; x < 2; ++x) {
            ui[x] = PREFILL ? 0 : uu[x] >> csh;
            uc[x] = PREFILL ? uu[x] : uu[x] & csh;
          }
          uint32_t r[2][16];
  #pragma unroll
          for (int x = 0; x < 2; ++x)
            if (uu[x] < nunits_g)
              tmem_ld16(tmem + lane_base + (uint32_t)(a * acc_cols + ui[x] * p.ncols + uc[x] * 16),
                        r[x]);
          tmem_ld_wait();
  #pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (uu[x] >= nunits_g) break;
            const int i = ui[x], c0 = uc[x] * 16;
            const int it = g * G + i;
            const int b = tile_seq(it);
            const int64_t j = (int64_t)tile_row0(it) + row;
            if (j >= p.E) continue;
            uint32_t sbits;
            if (scales_in_smem && NB == 2)
              sbits = *reinterpret_cast<const uint16_t*>(stiles + ring_tile(it) * kScaleTileBytes +
                                                         row * 2);
            else
              sbits = NB == 2
                  ? (uint32_t)*reinterpret_cast<const uint16_t*>(p.ki_scales + ((int64_t)b * p.E + j) * 2)
                  : (uint32_t)p.ki_scales[(int64_t)b * p.E + j];
            float sk[NB];
            sk[0] = exp2_int((int)(sbits & 0xFF) - 127);
            if (NB == 2) sk[NB - 1] = exp2_int((int)((sbits >> 8) & 0xFF) - 127);
            uint16_t* srow = p.scores + ((int64_t)b * p.Nq + i0) * p.E + j;
  #pragma unroll
            for (int cc = 0; cc < 16; cc += CPQ) {
              const int ql = (c0 + cc) / CPQ;
              if (ql < nq) {
                float sc = 0.f;
  #pragma unroll
                for (int h = 0; h < H_I; ++h) {
                  float dot = 0.f;
  #pragma unroll
                  for (int blk = 0; blk < NB; ++blk) {
                    const int c_in = cc + h * NB * SW + blk;                  // blocks in place
                    const int c_sw = cc + h * NB * SW + (SW - 1) * NB + blk;  // blocks swapped
                    const float d = swapped ? __uint_as_float(r[x][c_sw])
                                            : __uint_as_float(r[x][c_in]);
                    const float qm =
                        q_in_mma ? 1.f
                                 : exp2_int((int)qbyte[(b - b_first) * p.ncols + c0 + c_in] - 127);
                    dot = fmaf(d * qm, sk[blk], dot);
                  }
                  sc += fmaxf(dot, 0.f);
                }
                sc += 0.0f;  // -0 -> +0
                if (j < qvis[ql]) {
                  srow[(int64_t)ql * p.E] = f32_to_bf16_bits(sc);
                  if constexpr (F32OUT)
                    p.scores_f32[(srow - p.scores) + (int64_t)ql * p.E] = sc;
                }
              }
            }
          }
        }
      }
      if (PREFILL && sub == 0 && g + p.nacc < ntiles) {
        // this group's accumulator and scale region are free once this warp arrives: the
        // scales of the tile that reuses them go in first
        if (!write_sfa(g + p.nacc, a) && lane == 0) *aborted = 1;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[a]);
        // the slot's last group: its scale tile is no longer read by this warp
        if (unit_done) mbar_arrive(&empty[slot]);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(done);
  }

  // Teardown: tensor memory is freed by the allocating warp only after every epilogue warp has
  // signalled `done` (and the MMA warp has drained its MMAs above); the other warps just exit.
  __syncwarp();
  if (warp == 1) {
    mbar_wait_warp(done, 0, p.status, p.wait_budget);  // bounded; a timeout is already recorded
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

template <int H_I, int NB, int SW, bool PREFILL, bool F32OUT>
cudaError_t launch_t1(const CUtensorMap* kmap, const IdxParams& prm, const IndexerPlan& plan, int B,
                      cudaStream_t stream) {
  auto kern = indexer_kernel<H_I, NB, SW, PREFILL, F32OUT>;
  constexpr int EW = PREFILL ? 4 : 2;
  const size_t smem = smem_bytes((prm.Nq == 1 ? kMaxSeqPerCta : 1) * prm.ncols);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)plan.n_splits, (unsigned)plan.n_groups,
            (unsigned)(prm.Nq == 1 ? 1 : B));
  ProfScope prof(stream, "indexer_mxf4");
  return launch_ex(kern, grid, dim3(threads_for(EW)), smem, stream, 1, *kmap, prm);
}

template <int H_I, int NB, int SW, bool PREFILL>
cudaError_t launch_t(const CUtensorMap* kmap, const IdxParams& prm, const IndexerPlan& plan, int B,
                     cudaStream_t stream) {
  return prm.scores_f32 ? launch_t1<H_I, NB, SW, PREFILL, true>(kmap, prm, plan, B, stream)
                        : launch_t1<H_I, NB, SW, PREFILL, false>(kmap, prm, plan, B, stream);
}

int next_pow2_at_least32(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

}  // namespace

// Bulk-copy path: 32-byte key rows, each head doubled into 16 columns, 16-byte aligned scale runs.
bool indexer_bulk_path(int H_I, int d_I, int64_t E, int Nq) {
  return Nq == 1 && d_I == 64 && H_I <= 4 && E % 8 == 0;
}

IndexerPlan plan_indexer(int B, int Nq, int64_t E, int H_I, int d_I, bool paged) {
  IndexerPlan pl{};
  // paged keys are copied whole-tile from their pages: the bulk path whatever E is
  // prefill: one column per (query, head), both blocks scaled inside the MMA
  const int cpq = Nq > 1 ? H_I
                         : H_I * (d_I / 32) * (indexer_bulk_path(H_I, d_I, paged ? 8 : E, Nq) ? 2 : 1);
  if (Nq == 1) {  // two CTAs per SM: 3 x 64 + 32 scale columns fit in 256
    pl.QN = 1;
    pl.ncols = cpq > 16 ? 32 : 16;
    pl.G = kMaxG;
    pl.nacc = 3;
  } else {         // one CTA per SM: 2 x 224 + 3 x 16 scale columns fit in 512
    pl.QN = kMaxCols / cpq;
    pl.ncols = pl.QN * cpq;
    pl.G = 1;
    pl.nacc = 2;
  }
  pl.n_groups = (Nq + pl.QN - 1) / pl.QN;
  const int64_t tiles = (E + kTileM - 1) / kTileM;
  if (Nq == 1) {
    // persistent: two CTAs per SM over all (sequence, tile) pairs; a CTA spans at most
    // kMaxSeqPerCta sequences
    const int64_t total = (int64_t)B * tiles;
    int64_t g = (int64_t)kNumSMs * 2;
    const int64_t span_min = ((int64_t)B * tiles + (int64_t)(kMaxSeqPerCta - 1) * tiles - 1) /
                             ((int64_t)(kMaxSeqPerCta - 1) * tiles);
    if (g < span_min) g = span_min;
    if (g > total) g = total;
    pl.n_splits = (int)(g < 1 ? 1 : g);
  } else {
    const int64_t units = (int64_t)B * pl.n_groups;
    const int64_t target = (int64_t)kNumSMs;
    int64_t splits = (target + units - 1) / units;
    if (splits > tiles) splits = tiles;
    if (splits < 1) splits = 1;
    pl.n_splits = (int)splits;
  }
  pl.tmem_cols = next_pow2_at_least32(pl.nacc * pl.G * pl.ncols +
                                      (Nq > 1 ? pl.nacc + 1 : 2) * kSfCols);
  return pl;
}

cudaError_t launch_indexer(const CUtensorMap* kmap, const uint8_t* ki_codes, const uint8_t* qi_codes,
                           const uint8_t* qi_scales, const uint8_t* ki_scales, uint16_t* scores,
                           int B, int Nq, int64_t q_pos0, int64_t E, int m, int H_I, int d_I,
                           const IndexerPlan& plan, uint32_t* status, cudaStream_t stream,
                           float* scores_f32, const PagedLayout* paged, int64_t keys_fresh_from,
                           bool q_fresh) {
  IdxParams prm;
  prm.keys_fresh_from = keys_fresh_from;
  prm.q_fresh = q_fresh ? 1 : 0;
  const FaultConfig fc = fault_config();
  prm.wait_budget = fc.wait_budget;
  prm.fault_mask = fc.skip_mask;
  prm.block_table = paged ? paged->block_table : nullptr;
  prm.max_blocks = paged ? paged->max_blocks : 0;
  prm.n_pages = paged ? paged->n_pages : 0;
  prm.page_shift = 0;
  if (paged) {
    while ((1 << prm.page_shift) < kPageTokens / m) ++prm.page_shift;
    if (!indexer_bulk_path(H_I, d_I, 8, Nq) || (1 << prm.page_shift) % kTileM != 0)
      return cudaErrorInvalidValue;  // paged keys: decode bulk-copy path, whole tiles per page
  }
  prm.qi_codes = qi_codes;
  prm.qi_scales = qi_scales;
  prm.ki_scales = ki_scales;
  prm.scores = scores;
  prm.scores_f32 = scores_f32;
  prm.q_pos0 = q_pos0;
  prm.E = E;
  prm.Nq = Nq;
  prm.m = m;
  prm.QN = plan.QN;
  prm.ncols = plan.ncols;
  prm.G = plan.G;
  prm.nacc = plan.nacc;
  prm.n_splits = plan.n_splits;
  prm.tmem_cols = plan.tmem_cols;
  prm.B = B;
  prm.tiles_per_seq = (int)((E + kTileM - 1) / kTileM);
  prm.total_tiles = (int64_t)B * prm.tiles_per_seq;
  if (prm.total_tiles >= ((int64_t)1 << 31) || plan.n_splits >= (1 << 15))
    return cudaErrorInvalidValue;  // the decode range arithmetic is 32-bit
  prm.ki_codes = ki_codes;
  prm.status = status;
  const int NB = d_I / 32;
  const int SW = indexer_bulk_path(H_I, d_I, paged ? 8 : E, Nq) ? 2 : 1;
#define CSA_IDX_CASE(HH, NN, SS, PP)                                          \
  if (H_I == HH && NB == NN && SW == SS && prefill == PP)                     \
    return launch_t<HH, NN, SS, PP>(kmap, prm, plan, B, stream);
  const bool prefill = Nq > 1;
  CSA_IDX_CASE(1, 1, 1, false) CSA_IDX_CASE(2, 1, 1, false) CSA_IDX_CASE(4, 1, 1, false)
  CSA_IDX_CASE(8, 1, 1, false) CSA_IDX_CASE(1, 2, 2, false) CSA_IDX_CASE(2, 2, 2, false)
  CSA_IDX_CASE(4, 2, 2, false) CSA_IDX_CASE(8, 2, 1, false) CSA_IDX_CASE(1, 2, 1, false)
  CSA_IDX_CASE(2, 2, 1, false) CSA_IDX_CASE(4, 2, 1, false)
  CSA_IDX_CASE(1, 1, 1, true) CSA_IDX_CASE(2, 1, 1, true) CSA_IDX_CASE(4, 1, 1, true)
  CSA_IDX_CASE(8, 1, 1, true) CSA_IDX_CASE(8, 2, 1, true) CSA_IDX_CASE(1, 2, 1, true)
  CSA_IDX_CASE(2, 2, 1, true) CSA_IDX_CASE(4, 2, 1, true)
#undef CSA_IDX_CASE
  return cudaErrorInvalidValue;
}

}  // namespace csa
