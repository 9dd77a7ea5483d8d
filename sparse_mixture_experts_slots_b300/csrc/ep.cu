// Expert parallelism: regrouping of the rows an expert-owning rank receives (sm_103a).
//
// The Switch Transformers card (ai-papers.xuzou.cn, 方法适配) shards the experts over
// the cores and moves tokens with two all-to-alls around the expert FFN.  Here rank r owns a
// contiguous range of El experts; every source rank s sends it the blocks [El][R][d] of its
// dispatched buffer for those experts (fixed-size chunks, the first counts[s][e] rows of
// each block valid).  The receiver packs them per expert, source by source:
//     packed[e][off(s, e) + i] = chunk[s][e][i],  i < counts[s][e],
//     off(s, e) = sum over s' < s of counts[s'][e],
// so the expert FFN sees each local expert's rows contiguous; the inverse copy puts the
// expert outputs back into per-source chunks for the return all-to-all.
#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int EP_WARPS = 8;

// One warp per (source, expert, row) of the chunked layout.  rows_out (forward only, may
// be null): the packed row count of each local expert.  A count outside 0 .. R marks its
// block as holding no rows (every index then stays inside both buffers).
__global__ void __launch_bounds__(EP_WARPS * 32) ep_regroup_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                                   const int32_t* __restrict__ counts,
                                                                   int32_t* __restrict__ rows_out, int W, int El, int R,
                                                                   int vecs, int inverse) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long w = (long long)blockIdx.x * EP_WARPS + warp;
  if (rows_out && w < El && lane == 0) {
    int tot = 0;
    for (int s = 0; s < W; ++s) {
      const int c = counts[(size_t)s * El + (int)w];
      tot += (c < 0 || c > R) ? 0 : c;
    }
    rows_out[w] = tot;
  }
  if (w >= (long long)W * El * R) return;
  const int i = (int)(w % R);
  const int se = (int)(w / R);  // s * El + e
  const int s = se / El, e = se - s * El;
  const int n = counts[se];
  if (i >= n || n > R) return;  // n > R: a count no chunk can hold, nothing is copied
  long long off = 0;
  for (int sp = 0; sp < s; ++sp) {
    const int c = counts[(size_t)sp * El + e];
    off += (c < 0 || c > R) ? 0 : c;  // blocks with invalid counts hold no rows
  }
  if (off + i >= (long long)W * R) return;
  const long long chunk_row = (long long)se * R + i;
  const long long packed_row = (long long)e * W * R + off + i;
  const uint4* from = src + (inverse ? packed_row : chunk_row) * vecs;
  uint4* to = dst + (inverse ? chunk_row : packed_row) * vecs;
  for (int v = lane; v < vecs; v += 32) to[v] = __ldg(from + v);
}

int launch_ep_regroup(const void* src, void* dst, const int32_t* counts, int32_t* rows_out, int W, int El, int R,
                      int row_bytes, bool inverse, cudaStream_t s) {
  const long long rows = (long long)W * El * R;
  const long long warps = rows > El ? rows : El;
  if (warps == 0) return 0;
  const unsigned blocks = (unsigned)((warps + EP_WARPS - 1) / EP_WARPS);
  return launch_k(ep_regroup_kernel, dim3(blocks), dim3(EP_WARPS * 32), 0, s, false, 1, (const uint4*)src, (uint4*)dst,
                  counts, rows_out, W, El, R, row_bytes / 16, inverse ? 1 : 0) == cudaSuccess
             ? 1
             : -1;
}

}  // namespace smoe
