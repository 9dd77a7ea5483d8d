// Dispatch gather and combine scatter (sm_103a): rows staged through shared memory by 1-D
// TMA bulk copies (cp.async.bulk), 16-byte vectors where a warp touches a row itself.
//
// Dispatch: kept tokens are copied into their expert's block of xe; switch_dispatch also
// zeroes the rest of the block, as the one-hot dispatch tensor of the Switch Transformers
// card (ai-papers.xuzou.cn, 方法适配) would give.
// Combine: y_t = p_{e*}(x_t) * f_{e*}(x_t) for kept tokens and 0 for dropped ones
// ("042 · Switch Transformer：每个词只选一个专家", section 一; the gate is not
// renormalised, section 只执行一个专家时检查路由是否被错误归一化).
//
// Staging: each warp owns `bt` tokens' row slots of shared memory.  For a batch of up to bt
// tokens lane j issues the bulk loads (global -> shared) of token j's source rows into its
// slots, counted on the warp's mbarrier, and meanwhile works out where the token goes; after
// the wait lane j issues the bulk store (shared -> global) of its slot to the destination row
// and commits it as its own bulk group.  A slot is loaded again only after the lane's earlier
// stores have read it.  Zero fills are bulk stores from a zero row at the start of the CTA's
// shared memory.  One CTA per SM holds up to 192 KB of slots in flight.  Rows whose slots do
// not fit four warps (about 45 KB per token) take the register kernels below instead.
#include <algorithm>
#include <utility>

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

static int launch_dispatch_regs(const void* x, void* xe, const int32_t* expert, const int32_t* row,
                                const int32_t* expert2, const int32_t* row2, const int32_t* expert_rows, int N,
                                int E, int R, int row_bytes, cudaStream_t s) {
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

static int launch_dispatch_slots_regs(const void* x, void* xe, const RouteArgs& a, void* y, const void* resid,
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

static int launch_combine_regs(const void* ye, const int32_t* expert, const int32_t* row, const float* gate,
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

// ---------------------------------------------------------------- TMA-staged kernels
constexpr int BULK_SLOT_BYTES = 192 * 1024;  // row slots of one CTA
constexpr int BULK_SMEM_MAX = 226 * 1024;    // dynamic shared memory of one CTA, at most
constexpr int BULK_MAX_WARPS = 16;
constexpr int BULK_MIN_WARPS = 4;

struct BulkPlan {
  bool ok = false;
  int warps = 0, bt = 0, ctas = 0;
  long long batches = 0;  // token batches of bt tokens
  size_t smem = 0;
};

// Shared memory of a staging CTA: the zero row (rounded up to 128 bytes), one mbarrier per
// warp (128 bytes), then warps x bt x rpt row slots.
__host__ __device__ inline int bulk_zero_bytes(int row_bytes) { return (row_bytes + 127) & ~127; }

// items tokens with rpt rows of row_bytes each.  Tokens per batch shrink (down to 1) until
// the batches cover every SM's warps once.
static BulkPlan bulk_plan(long long items, int row_bytes, int rpt) {
  BulkPlan p;
  const long long tok_bytes = (long long)row_bytes * rpt;
  if (row_bytes <= 0 || row_bytes % 16 != 0) return p;
  const long long budget = std::min<long long>(BULK_SLOT_BYTES, BULK_SMEM_MAX - bulk_zero_bytes(row_bytes) - 128);
  if (tok_bytes * BULK_MIN_WARPS > budget) return p;
  p.warps = (int)std::min<long long>(BULK_MAX_WARPS, budget / tok_bytes);
  const int bt_max = (int)std::min<long long>(32, budget / (tok_bytes * p.warps));
  const long long sms = device_sm_count();
  const long long want = (items + sms * p.warps - 1) / (sms * p.warps);
  p.bt = (int)std::max<long long>(1, std::min<long long>(bt_max, want));
  p.batches = (items + p.bt - 1) / p.bt;
  p.smem = (size_t)bulk_zero_bytes(row_bytes) + 128 + (size_t)p.warps * p.bt * tok_bytes;
  p.ok = true;
  return p;
}

// The CTA prologue of every staging kernel: zero row, one mbarrier per warp, both visible
// to the async proxy before any bulk copy uses them.
__device__ __forceinline__ uint64_t* bulk_prologue(uint8_t* bsm, int row_bytes) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int i = threadIdx.x; i < row_bytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(bsm)[i] = make_uint4(0, 0, 0, 0);
  uint64_t* bar = reinterpret_cast<uint64_t*>(bsm + bulk_zero_bytes(row_bytes)) + warp;
  if (lane == 0) mbar_init(bar, 1);
  fence_mbar_init();
  fence_proxy_async_smem();
  __syncthreads();
  return bar;
}

// Forward path: the slots of the routing step and the dispatch copy in one pass, rows
// staged by bulk copies.  Lane j of a batch loads token j's row while it turns the token's
// in-tile rank (held in slot[]) into its slot, keep flag and row (as route_slots_kernel
// does); the slot then goes to the expert block, or, for a dropped token with the combine
// fused into the FFN, y gets zero (a store from the zero row) or the residual (plain 16-byte
// copies).  Rows of an expert block past its count are left as they are: the forward's
// expert FFN never uses them.
__global__ void __launch_bounds__(BULK_MAX_WARPS * 32) dispatch_slots_bulk_kernel(
    const uint8_t* __restrict__ x, uint8_t* __restrict__ xe, const int32_t* __restrict__ expert,
    const int32_t* __restrict__ tile_base, const int32_t* __restrict__ group_off, int32_t* __restrict__ slot,
    uint8_t* __restrict__ keep, int32_t* __restrict__ row, int32_t* __restrict__ tok_of_row, long long N, int T,
    int E, int nT, int C, int R, int row_bytes, int bt, long long batches, bool debug, uint32_t* err,
    uint8_t* __restrict__ y, const uint8_t* __restrict__ resid, uint32_t* __restrict__ zero_ptr, int zero_words) {
  extern __shared__ __align__(128) uint8_t bsm[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  uint64_t* bar = bulk_prologue(bsm, row_bytes);
  uint8_t* my = bsm + bulk_zero_bytes(row_bytes) + 128 + ((size_t)warp * bt + lane) * row_bytes;
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zero_ptr[i] = 0u;
  uint32_t phase = 0;
  bool ok = true;
  for (long long b = (long long)blockIdx.x * nw + warp; b < batches; b += (long long)gridDim.x * nw) {
    const long long w = b * bt + lane;
    const int nb = (int)min((long long)bt, N - b * bt);
    bulk_wait_read_all();  // this lane's earlier store has read its slot
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)nb * (uint32_t)row_bytes);
    __syncwarp();
    if (lane < nb) bulk_load(my, x + w * row_bytes, (uint32_t)row_bytes, bar);
    int r = -1, e = 0;
    if (lane < nb) {
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
    if (!__all_sync(0xffffffffu, mbar_wait(bar, phase))) {
      ok = false;
      break;
    }
    phase ^= 1u;
    if (lane < nb) {
      if (r >= 0) {
        bulk_store(xe + ((size_t)e * R + r) * row_bytes, my, (uint32_t)row_bytes);
        bulk_commit();
      } else if (y && !resid) {  // a dropped token skips the expert: y is zero
        bulk_store(y + w * row_bytes, bsm, (uint32_t)row_bytes);
        bulk_commit();
      }
    }
    if (y && resid) {  // ... or the residual alone
      unsigned m = __ballot_sync(0xffffffffu, lane < nb && r < 0);
      while (m) {
        const int j = __ffs(m) - 1;
        m &= m - 1;
        const uint4* src = reinterpret_cast<const uint4*>(resid + (b * bt + j) * row_bytes);
        uint4* dst = reinterpret_cast<uint4*>(y + (b * bt + j) * row_bytes);
        for (int k = lane; k < row_bytes / 16; k += 32) dst[k] = __ldg(src + k);
      }
    }
  }
  if (!ok) {
    raise_error(err, ERR_TIMEOUT);
    mbar_wait(bar, phase);  // bounded again: the batch's loads in flight
  }
  bulk_wait_read_all();  // the stores read their slots before the CTA leaves; the writes finish with the grid
}

// switch_dispatch and the unfused forward: batches [0, tok_batches) copy kept tokens' rows
// to their first (and, top-2, second) choice's block; batches past them zero 32 rows each
// of the expert blocks past their counts (stores from the zero row).
__global__ void __launch_bounds__(BULK_MAX_WARPS * 32) dispatch_bulk_kernel(
    const uint8_t* __restrict__ x, uint8_t* __restrict__ xe, const int32_t* __restrict__ expert,
    const int32_t* __restrict__ row, const int32_t* __restrict__ expert2, const int32_t* __restrict__ row2,
    const int32_t* __restrict__ expert_rows, long long N, int E, int R, int row_bytes, int bt, long long tok_batches,
    long long batches, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t bsm[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  uint64_t* bar = bulk_prologue(bsm, row_bytes);
  uint8_t* my = bsm + bulk_zero_bytes(row_bytes) + 128 + ((size_t)warp * bt + lane) * row_bytes;
  griddep_wait();
  griddep_launch_dependents();
  uint32_t phase = 0;
  bool ok = true;
  for (long long b = (long long)blockIdx.x * nw + warp; b < batches; b += (long long)gridDim.x * nw) {
    if (b >= tok_batches) {
      const long long dr = (b - tok_batches) * 32 + lane;
      if (dr < (long long)E * R) {
        const int e = (int)(dr / R), r = (int)(dr % R);
        if (r >= expert_rows[e]) {
          bulk_store(xe + dr * row_bytes, bsm, (uint32_t)row_bytes);
          bulk_commit();
        }
      }
      continue;
    }
    const long long w = b * bt + lane;
    const int nb = (int)min((long long)bt, N - b * bt);
    int r = -1, r2 = -1, e = 0, e2 = 0;
    if (lane < nb) {  // records outside the blocks are reported and skipped
      r = row[w];
      if (r >= 0) e = expert[w];
      if (r >= R || e < 0 || e >= E) {
        raise_error(err, ERR_BOUNDS);
        r = -1;
      }
      if (row2) {
        r2 = row2[w];
        if (r2 >= 0) e2 = expert2[w];
        if (r2 >= R || e2 < 0 || e2 >= E) {
          raise_error(err, ERR_BOUNDS);
          r2 = -1;
        }
      }
    }
    const bool load = r >= 0 || r2 >= 0;
    const unsigned nload = __popc(__ballot_sync(0xffffffffu, load));
    bulk_wait_read_all();
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, nload * (uint32_t)row_bytes);
    __syncwarp();
    if (load) bulk_load(my, x + w * row_bytes, (uint32_t)row_bytes, bar);
    if (!__all_sync(0xffffffffu, mbar_wait(bar, phase))) {
      ok = false;
      break;
    }
    phase ^= 1u;
    if (load) {
      if (r >= 0) bulk_store(xe + ((size_t)e * R + r) * row_bytes, my, (uint32_t)row_bytes);
      if (r2 >= 0) bulk_store(xe + ((size_t)e2 * R + r2) * row_bytes, my, (uint32_t)row_bytes);
      bulk_commit();
    }
  }
  if (!ok) {
    raise_error(err, ERR_TIMEOUT);
    mbar_wait(bar, phase);
  }
  bulk_wait_read_all();  // the stores read their slots before the CTA leaves; the writes finish with the grid
}

// Combine with staged rows: lane j loads token j's expert output row(s) and its residual row
// into its slots; after the wait the warp computes each token's y row in place in its first
// slot (same arithmetic as combine_kernel) and lane j stores it.  A token with no kept choice
// stores the residual slot, or the zero row.
template <bool BF16>
__global__ void __launch_bounds__(BULK_MAX_WARPS * 32) combine_bulk_kernel(
    const uint8_t* __restrict__ ye, const int32_t* __restrict__ expert, const int32_t* __restrict__ row,
    const float* __restrict__ gate, const int32_t* __restrict__ expert2, const int32_t* __restrict__ row2,
    const float* __restrict__ gate2, const uint8_t* __restrict__ resid, uint8_t* __restrict__ y, long long N, int E,
    int R, int row_bytes, int bt, int rpt, long long batches, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t bsm[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  uint64_t* bar = bulk_prologue(bsm, row_bytes);
  uint8_t* wslots = bsm + bulk_zero_bytes(row_bytes) + 128 + (size_t)warp * bt * rpt * row_bytes;
  uint8_t* my = wslots + (size_t)lane * rpt * row_bytes;  // [first, second (top-2), residual]
  const int k2 = 1, kres = expert2 ? 2 : 1;
  const int vecs = row_bytes / 16;
  griddep_wait();
  griddep_launch_dependents();
  uint32_t phase = 0;
  bool ok = true;
  for (long long b = (long long)blockIdx.x * nw + warp; b < batches; b += (long long)gridDim.x * nw) {
    const long long t = b * bt + lane;
    const int nb = (int)min((long long)bt, N - b * bt);
    int r = -1, r2 = -1, e = 0, e2 = 0;
    float g = 0.f, g2 = 0.f;
    if (lane < nb) {  // records outside the blocks are reported and count as dropped
      r = row[t];
      if (r >= 0) e = expert[t];
      if (r >= R || e < 0 || e >= E) {
        raise_error(err, ERR_BOUNDS);
        r = -1;
      }
      if (r >= 0) g = gate[t];
      if (expert2) {
        r2 = row2[t];
        if (r2 >= 0) e2 = expert2[t];
        if (r2 >= R || e2 < 0 || e2 >= E) {
          raise_error(err, ERR_BOUNDS);
          r2 = -1;
        }
        if (r2 >= 0) g2 = gate2[t];
      }
    }
    const uint32_t rows = (r >= 0) + (r2 >= 0) + (resid && lane < nb ? 1 : 0);
    const uint32_t total = __reduce_add_sync(0xffffffffu, rows);
    bulk_wait_read_all();
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(bar, total * (uint32_t)row_bytes);
    __syncwarp();
    if (r >= 0) bulk_load(my, ye + ((size_t)e * R + r) * row_bytes, (uint32_t)row_bytes, bar);
    if (r2 >= 0) bulk_load(my + k2 * row_bytes, ye + ((size_t)e2 * R + r2) * row_bytes, (uint32_t)row_bytes, bar);
    if (resid && lane < nb) bulk_load(my + kres * row_bytes, resid + t * row_bytes, (uint32_t)row_bytes, bar);
    if (!__all_sync(0xffffffffu, mbar_wait(bar, phase))) {
      ok = false;
      break;
    }
    phase ^= 1u;
    for (int j = 0; j < nb; ++j) {
      const int rj = __shfl_sync(0xffffffffu, r, j), r2j = __shfl_sync(0xffffffffu, r2, j);
      const float gj = __shfl_sync(0xffffffffu, g, j), g2j = __shfl_sync(0xffffffffu, g2, j);
      if (rj < 0 && r2j < 0) continue;  // stored straight from the residual slot or the zero row
      uint4* s0 = reinterpret_cast<uint4*>(wslots + (size_t)j * rpt * row_bytes);
      const uint4* s1 = s0 + k2 * vecs;
      const uint4* sr = s0 + kres * vecs;
      for (int v = lane; v < vecs; v += 32) {
        constexpr int W = BF16 ? 8 : 4;
        float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (rj >= 0) {
          const uint4 in = s0[v];
          if (BF16) {
            unpack8(in, o);
          } else {
            const float* f = reinterpret_cast<const float*>(&in);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = f[i];
          }
#pragma unroll
          for (int i = 0; i < W; ++i) o[i] *= gj;
        }
        if (r2j >= 0) {
          float o2[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          const uint4 in = s1[v];
          if (BF16) {
            unpack8(in, o2);
          } else {
            const float* f = reinterpret_cast<const float*>(&in);
#pragma unroll
            for (int i = 0; i < 4; ++i) o2[i] = f[i];
          }
#pragma unroll
          for (int i = 0; i < W; ++i) o[i] = fmaf(g2j, o2[i], o[i]);
        }
        if (resid) {
          const uint4 rv = sr[v];
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
        s0[v] = BF16 ? pack8(o)
                     : make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                                  __float_as_uint(o[3]));
      }
    }
    fence_proxy_async_smem();  // the y rows written above, before the bulk stores read them
    __syncwarp();
    if (lane < nb) {
      const uint8_t* src = (r >= 0 || r2 >= 0) ? my : (resid ? my + kres * row_bytes : bsm);
      bulk_store(y + t * row_bytes, src, (uint32_t)row_bytes);
      bulk_commit();
    }
  }
  if (!ok) {
    raise_error(err, ERR_TIMEOUT);
    mbar_wait(bar, phase);
  }
  bulk_wait_read_all();  // the stores read their slots before the CTA leaves; the writes finish with the grid
}

template <typename K, typename... Args>
static int launch_bulk(K kern, const BulkPlan& p, cudaStream_t s, bool pdl, Args&&... args) {
  // the plans' bound, not this plan's size: one value whatever the shape, so calls from
  // several host threads never lower it under one another's launch
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, BULK_SMEM_MAX) != cudaSuccess) return -1;
  return launch_k(kern, dim3((unsigned)p.ctas), dim3((unsigned)p.warps * 32), p.smem, s, pdl, 1,
                  std::forward<Args>(args)...) == cudaSuccess
             ? 1
             : -1;
}

static long long bulk_ctas(long long batches, int warps) {
  const long long want = (batches + warps - 1) / warps;
  const long long sms = device_sm_count();
  return std::max<long long>(1, std::min<long long>(want, sms));
}

int launch_dispatch_slots(const void* x, void* xe, const RouteArgs& a, void* y, const void* resid,
                          uint32_t* zero_ptr, int zero_words, cudaStream_t s, bool pdl) {
  const long long N = (long long)a.G * a.T;
  const int row_bytes = a.d * (a.x_bf16 ? 2 : 4);
  BulkPlan p = bulk_plan(N, row_bytes, 1);
  if (!p.ok) return launch_dispatch_slots_regs(x, xe, a, y, resid, zero_ptr, zero_words, s, pdl);
  if (N == 0 && zero_words == 0) return 0;
  p.ctas = (int)bulk_ctas(p.batches, p.warps);
  const int nT = (a.T + ROUTE_TILE - 1) / ROUTE_TILE;
  return launch_bulk(dispatch_slots_bulk_kernel, p, s, pdl, (const uint8_t*)x, (uint8_t*)xe, a.expert, a.tile_base,
                     a.group_off, a.slot, a.keep, a.row, a.tok_of_row, N, a.T, a.E, nT, a.C, a.R, row_bytes, p.bt,
                     p.batches, a.debug, a.err, (uint8_t*)y, (const uint8_t*)resid, zero_ptr, zero_words);
}

int launch_dispatch(const void* x, void* xe, const int32_t* expert, const int32_t* row, const int32_t* expert2,
                    const int32_t* row2, const int32_t* expert_rows, int N, int E, int R, int row_bytes,
                    uint32_t* err, cudaStream_t s) {
  if ((long long)E * R == 0) return 0;
  BulkPlan p = bulk_plan(N, row_bytes, 1);
  if (!p.ok) return launch_dispatch_regs(x, xe, expert, row, expert2, row2, expert_rows, N, E, R, row_bytes, s);
  const long long zb = ((long long)E * R + 31) / 32;
  const long long batches = p.batches + zb;
  p.ctas = (int)bulk_ctas(batches, p.warps);
  return launch_bulk(dispatch_bulk_kernel, p, s, false, (const uint8_t*)x, (uint8_t*)xe, expert, row, expert2, row2,
                     expert_rows, (long long)N, E, R, row_bytes, p.bt, p.batches, batches, err);
}

int launch_combine(const void* ye, const int32_t* expert, const int32_t* row, const float* gate,
                   const int32_t* expert2, const int32_t* row2, const float* gate2, const void* resid,
                   void* y, int N, int d, int E, int R, bool bf16, uint32_t* err, cudaStream_t s, bool pdl) {
  if (N == 0) return 0;
  const int row_bytes = d * (bf16 ? 2 : 4);
  const int rpt = 1 + (expert2 ? 1 : 0) + (resid ? 1 : 0);
  BulkPlan p = bulk_plan(N, row_bytes, rpt);
  if (!p.ok)
    return launch_combine_regs(ye, expert, row, gate, expert2, row2, gate2, resid, y, N, d, R, bf16, s, pdl);
  p.ctas = (int)bulk_ctas(p.batches, p.warps);
  if (bf16)
    return launch_bulk(combine_bulk_kernel<true>, p, s, pdl, (const uint8_t*)ye, expert, row, gate, expert2, row2,
                       gate2, (const uint8_t*)resid, (uint8_t*)y, (long long)N, E, R, row_bytes, p.bt, rpt,
                       p.batches, err);
  return launch_bulk(combine_bulk_kernel<false>, p, s, pdl, (const uint8_t*)ye, expert, row, gate, expert2, row2,
                     gate2, (const uint8_t*)resid, (uint8_t*)y, (long long)N, E, R, row_bytes, p.bt, rpt, p.batches,
                     err);
}

}  // namespace smoe
