// Batched row copies on the device, for a serving loop's per-step inputs: the step's new rows
// (queries, index queries, the raw K/V rows, logits and index keys of the tokens it appends)
// arrive in one packed host-to-device copy into a staging buffer, and this one launch places
// them into the layer buffers, whose rows are strided by the sequence length.
#include <algorithm>

#include "kernels.h"
#include "prof.h"

namespace csa {
namespace {

struct ScatterParams {
  ScatterCopy c[kMaxScatterCopies];
};

constexpr int kSegBytes = 2048;  // bytes one warp moves per work item: 4 x 16 bytes per lane
constexpr int kWarps = 8;

// blockIdx.y: the copy. Its work items are (row, 2 KB segment of the row) pairs, taken by the
// grid's warps in turn; a warp's lanes move 16-byte pieces (four loads in flight, then four
// stores) when the copy is 16-byte aligned, else single bytes. The kernel does not signal
// dependents early: the launch after it (the layer's first kernel, which may read its inputs
// before its own grid-dependency wait) starts only once every row is in place.
__global__ void __launch_bounds__(32 * kWarps) scatter_rows_kernel(const ScatterParams p) {
  const ScatterCopy& c = p.c[blockIdx.y];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool vec = ((reinterpret_cast<uintptr_t>(c.dst) | reinterpret_cast<uintptr_t>(c.src) |
                     (uintptr_t)c.row_bytes | (uintptr_t)c.dst_stride) & 15u) == 0;
  const int64_t segs = (c.row_bytes + kSegBytes - 1) / kSegBytes;
  const int64_t items = c.rows * segs;
  for (int64_t it = (int64_t)blockIdx.x * kWarps + warp; it < items;
       it += (int64_t)gridDim.x * kWarps) {
    const int64_t r = segs == 1 ? it : it / segs;
    const int64_t b0 = (it - r * segs) * kSegBytes;
    const int64_t b1 = b0 + kSegBytes < c.row_bytes ? b0 + kSegBytes : c.row_bytes;
    const uint8_t* s = static_cast<const uint8_t*>(c.src) + r * c.row_bytes;
    uint8_t* d = static_cast<uint8_t*>(c.dst) + r * c.dst_stride;
    if (vec) {
      const int64_t x0 = (b0 >> 4) + lane, x1 = b1 >> 4;
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (x0 + 32 * k < x1) v[k] = reinterpret_cast<const uint4*>(s)[x0 + 32 * k];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (x0 + 32 * k < x1) reinterpret_cast<uint4*>(d)[x0 + 32 * k] = v[k];
    } else {
      for (int64_t x = b0 + lane; x < b1; x += 32) d[x] = s[x];
    }
  }
}

}  // namespace

cudaError_t launch_scatter_rows(const ScatterCopy* copies, int n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  ScatterParams prm = {};
  int64_t max_items = 0;
  for (int i = 0; i < n; ++i) {
    prm.c[i] = copies[i];
    max_items = std::max<int64_t>(
        max_items, copies[i].rows * ((copies[i].row_bytes + kSegBytes - 1) / kSegBytes));
  }
  const int64_t blocks = std::min<int64_t>((max_items + kWarps - 1) / kWarps, 4 * kNumSMs);
  if (blocks == 0) return cudaSuccess;
  ProfScope prof(stream, "scatter_rows");
  scatter_rows_kernel<<<dim3((unsigned)blocks, (unsigned)n), 32 * kWarps, 0, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace csa
