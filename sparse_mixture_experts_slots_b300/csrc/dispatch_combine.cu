// Dispatch gather and combine scatter (sm_103a), 16-byte vectors.
//
// Dispatch: kept tokens are copied into their expert's block of xe; switch_dispatch also
// zeroes the rest of the block, as the one-hot dispatch tensor of the Switch Transformers
// card (ai-papers.xuzou.cn, 方法适配) would give.
// Combine: y_t = p_{e*}(x_t) * f_{e*}(x_t) for kept tokens and 0 for dropped ones
// ("042 · Switch Transformer：每个词只选一个专家", section 一; the gate is not
// renormalised, section 只执行一个专家时检查路由是否被错误归一化).
#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int DC_WARPS = 8;

// Warps [0, N) copy token rows to their slots; warps [N, N + E*R) zero the rows
// past each expert's count.  Both reads and writes are whole 16-byte-vector rows.
// expert2 / row2 (top-2 routing, else null): the token's second choice, copied from the
// same read of its row.
__global__ void __launch_bounds__(DC_WARPS * 32) dispatch_kernel(const uint4* __restrict__ x, uint4* __restrict__ xe,
                                                                 const int32_t* __restrict__ expert,
                                                                 const int32_t* __restrict__ row,
                                                                 const int32_t* __restrict__ expert2,
                                                                 const int32_t* __restrict__ row2,
                                                                 const int32_t* __restrict__ expert_rows, int N,
                                                                 int E, int R, int vecs) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long w = (long long)blockIdx.x * DC_WARPS + warp;
  if (w < N) {
    const int r = row[w];
    const int r2 = row2 ? row2[w] : -1;
    if (r < 0 && r2 < 0) return;
    const uint4* src = x + w * vecs;
    uint4* dst = r >= 0 ? xe + ((long long)expert[w] * R + r) * vecs : nullptr;
    uint4* dst2 = r2 >= 0 ? xe + ((long long)expert2[w] * R + r2) * vecs : nullptr;
    for (int v = lane; v < vecs; v += 32) {
      const uint4 val = __ldg(src + v);
      if (dst) dst[v] = val;
      if (dst2) dst2[v] = val;
    }
    return;
  }
  const long long dr = w - N;
  if (dr >= (long long)E * R) return;
  const int e = (int)(dr / R), r = (int)(dr % R);
  if (r < expert_rows[e]) return;
  uint4* dst = xe + dr * vecs;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int v = lane; v < vecs; v += 32) dst[v] = zero;
}

int launch_dispatch(const void* x, void* xe, const int32_t* expert, const int32_t* row, const int32_t* expert2,
                    const int32_t* row2, const int32_t* expert_rows, int N, int E, int R, int row_bytes, cudaStream_t s) {
  const long long warps = (long long)N + (long long)E * R;
  if (warps == 0 || (long long)E * R == 0) return 0;
  const unsigned blocks = (unsigned)((warps + DC_WARPS - 1) / DC_WARPS);
  return launch_k(dispatch_kernel, dim3(blocks), dim3(DC_WARPS * 32), 0, s, false, 1, (const uint4*)x, (uint4*)xe,
                  expert, row, expert2, row2, expert_rows, N, E, R, row_bytes / 16) == cudaSuccess
             ? 1
             : -1;
}

// Forward path: the slots of the routing step and the dispatch copy in one pass.
// Warp w takes tokens DS_TPW w .. DS_TPW w + DS_TPW - 1: every lane first loads its part of
// all of their rows (those reads do not depend on routing), while lane j < DS_TPW turns
// token j's in-tile rank (held in slot[]) into its slot, keep flag and row (as
// route_slots_kernel does); then each row goes to its expert block, or, for a dropped token
// with the combine fused into the FFN, y gets the residual (or zero).  Rows of an expert
// block past its count are left as they are: the forward's expert FFN never uses them (its
// MMA columns past a chunk's filled rows are discarded), unlike switch_dispatch's output.
constexpr int DS_VMAX = 4;  // 16-byte vectors per lane and row held in registers (rows <= 2 KB)
constexpr int DS_TPW = 4;   // tokens per warp

__global__ void __launch_bounds__(DC_WARPS * 32) dispatch_slots_kernel(
    const uint4* __restrict__ x, uint4* __restrict__ xe, const int32_t* __restrict__ expert,
    const int32_t* __restrict__ tile_base, const int32_t* __restrict__ group_off,
    int32_t* __restrict__ slot, uint8_t* __restrict__ keep, int32_t* __restrict__ row,
    int32_t* __restrict__ tok_of_row, long long N, int T, int E, int nT, int C, int R, int vecs, bool debug,
    uint32_t* err, uint4* __restrict__ y, const uint4* __restrict__ resid, uint32_t* __restrict__ zero_ptr,
    int zero_words) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long w0 = ((long long)blockIdx.x * DC_WARPS + warp) * DS_TPW;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zero_ptr[i] = 0u;
  if (w0 >= N) return;
  const bool in_regs = vecs <= 32 * DS_VMAX;
  uint4 v[DS_TPW][DS_VMAX];
  if (in_regs) {
#pragma unroll
    for (int j = 0; j < DS_TPW; ++j)
#pragma unroll
      for (int k = 0; k < DS_VMAX; ++k)
        if (w0 + j < N && lane + 32 * k < vecs) v[j][k] = __ldg(x + (w0 + j) * vecs + lane + 32 * k);
  }
  int r = -1, e = 0;
  if (lane < DS_TPW && w0 + lane < N) {
    const long long w = w0 + lane;
    const int g = (int)(w / T);
    const int ti = (int)(w - (long long)g * T);
    const int rank = slot[w];
    e = expert[w];
    if (e < 0 || e >= E) {
      raise_error(err, ERR_BOUNDS);
      e = 0;
      slot[w] = 0;
      keep[w] = 0;
    } else {
      const int s = tile_base[((size_t)g * nT + ti / ROUTE_TILE) * E + e] + rank;
      const int goff = group_off[(size_t)g * E + e];
      slot[w] = s;
      if (s < C) {
        r = goff + s;
        if (r < 0 || r >= R) {
          if (debug) raise_error(err, ERR_BOUNDS);
          r = -1;
        } else {
          tok_of_row[(size_t)e * R + r] = (int32_t)w;
        }
      }
      keep[w] = r >= 0 ? 1 : 0;
    }
    row[w] = r;
  }
#pragma unroll
  for (int j = 0; j < DS_TPW; ++j) {
    const int rj = __shfl_sync(0xffffffffu, r, j);
    const int ej = __shfl_sync(0xffffffffu, e, j);
    const long long w = w0 + j;
    if (w >= N) break;
    if (rj < 0) {
      if (y) {  // a dropped token skips the expert: y is the residual alone, or zero
        const uint4 zero = make_uint4(0, 0, 0, 0);
        for (int k = lane; k < vecs; k += 32) y[w * vecs + k] = resid ? __ldg(resid + w * vecs + k) : zero;
      }
      continue;
    }
    uint4* dst = xe + ((long long)ej * R + rj) * vecs;
    if (in_regs) {
#pragma unroll
      for (int k = 0; k < DS_VMAX; ++k)
        if (lane + 32 * k < vecs) dst[lane + 32 * k] = v[j][k];
    } else {
      for (int k = lane; k < vecs; k += 32) dst[k] = __ldg(x + w * vecs + k);
    }
  }
}

int launch_dispatch_slots(const void* x, void* xe, const RouteArgs& a, void* y, const void* resid,
                          uint32_t* zero_ptr, int zero_words, cudaStream_t s, bool pdl) {
  const long long N = (long long)a.G * a.T;
  long long warps = (N + DS_TPW - 1) / DS_TPW;
  if (warps == 0 && zero_words == 0) return 0;
  if (warps == 0) warps = 1;  // one block still clears the words
  const int nT = (a.T + ROUTE_TILE - 1) / ROUTE_TILE;
  const int vecs = a.d * (a.x_bf16 ? 2 : 4) / 16;
  const unsigned blocks = (unsigned)((warps + DC_WARPS - 1) / DC_WARPS);
  return launch_k(dispatch_slots_kernel, dim3(blocks), dim3(DC_WARPS * 32), 0, s, pdl, 1, (const uint4*)x, (uint4*)xe,
                  a.expert, a.tile_base, a.group_off, a.slot, a.keep, a.row, a.tok_of_row, N, a.T, a.E, nT, a.C, a.R,
                  vecs, a.debug, a.err, (uint4*)y, (const uint4*)resid, zero_ptr, zero_words) == cudaSuccess
             ? 1
             : -1;
}

// ---------------------------------------------------------------- combine
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __bfloat1622float2(h[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 v;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return v;
}

// expert2 / row2 / gate2 (top-2 routing, else null): y_t also gets gate2_t * ye of the
// token's second choice when that choice was kept.
template <bool BF16>
__global__ void __launch_bounds__(DC_WARPS * 32) combine_kernel(const uint4* __restrict__ ye,
                                                                const int32_t* __restrict__ expert,
                                                                const int32_t* __restrict__ row,
                                                                const float* __restrict__ gate,
                                                                const int32_t* __restrict__ expert2,
                                                                const int32_t* __restrict__ row2,
                                                                const float* __restrict__ gate2,
                                                                const uint4* __restrict__ resid, uint4* __restrict__ y,
                                                                int N, int R, int vecs) {
  griddep_wait();
  griddep_launch_dependents();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const long long t = (long long)blockIdx.x * DC_WARPS + warp;
  if (t >= N) return;
  const int r = row[t];
  const uint4* src = nullptr;
  float g = 0.f;
  if (r >= 0) {
    src = ye + ((long long)expert[t] * R + r) * vecs;
    g = gate[t];
  }
  const int r2 = row2 ? row2[t] : -1;
  const uint4* src2 = nullptr;
  float g2 = 0.f;
  if (r2 >= 0) {
    src2 = ye + ((long long)expert2[t] * R + r2) * vecs;
    g2 = gate2[t];
  }
  uint4* dst = y + t * vecs;
  const uint4* res = resid ? resid + t * vecs : nullptr;
  for (int v = lane; v < vecs; v += 32) {
    constexpr int W = BF16 ? 8 : 4;
    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (src) {
      const uint4 in = __ldg(src + v);
      if (BF16) {
        unpack8(in, o);
      } else {
        const float* f = reinterpret_cast<const float*>(&in);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = f[i];
      }
#pragma unroll
      for (int i = 0; i < W; ++i) o[i] *= g;
    }
    if (src2) {
      float o2[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      const uint4 in = __ldg(src2 + v);
      if (BF16) {
        unpack8(in, o2);
      } else {
        const float* f = reinterpret_cast<const float*>(&in);
#pragma unroll
        for (int i = 0; i < 4; ++i) o2[i] = f[i];
      }
#pragma unroll
      for (int i = 0; i < W; ++i) o[i] = fmaf(g2, o2[i], o[i]);
    }
    if (res) {
      const uint4 rv = __ldg(res + v);
      if (BF16) {
        float rf[8];
        unpack8(rv, rf);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] += rf[i];
      } else {
        const float* f = reinterpret_cast<const float*>(&rv);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] += f[i];
      }
    }
    if (BF16) {
      dst[v] = pack8(o);
    } else {
      dst[v] = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                          __float_as_uint(o[3]));
    }
  }
}

int launch_combine(const void* ye, const int32_t* expert, const int32_t* row, const float* gate,
                   const int32_t* expert2, const int32_t* row2, const float* gate2, const void* resid,
                   void* y, int N, int d, int R, bool bf16, cudaStream_t s, bool pdl) {
  if (N == 0) return 0;
  const int vecs = d * (bf16 ? 2 : 4) / 16;
  const unsigned blocks = (unsigned)((N + DC_WARPS - 1) / DC_WARPS);
  const cudaError_t e =
      bf16 ? launch_k(combine_kernel<true>, dim3(blocks), dim3(DC_WARPS * 32), 0, s, pdl, 1, (const uint4*)ye, expert,
                      row, gate, expert2, row2, gate2, (const uint4*)resid, (uint4*)y, N, R, vecs)
           : launch_k(combine_kernel<false>, dim3(blocks), dim3(DC_WARPS * 32), 0, s, pdl, 1, (const uint4*)ye, expert,
                      row, gate, expert2, row2, gate2, (const uint4*)resid, (uint4*)y, N, R, vecs);
  return e == cudaSuccess ? 1 : -1;
}

}  // namespace smoe
