// Routing kernels of the top-1 Switch layer (sm_103a).
//
// Stages, following the pipeline of "042 · Switch Transformer：每个词只选一个专家",
// section 三 (float32 router -> one expert per token -> load statistics and aux
// loss -> capacity truncation):
//   1. router_logits:   z = x W_r^T + b_r in float32 (x cast up; selective precision,
//                        Switch Transformers card on ai-papers.xuzou.cn, 方法适配).
//   2. route_softmax:   per token max/argmax (ties -> lowest index), softmax sum, gate;
//                        per 128-token tile: expert histogram and probability sums.
//   3. route_scan:      per (group, expert): exclusive prefix of tile histograms,
//                        raw and accepted counts, mean probability P.
//   4. route_finalize:  per group balance E * sum f P and aux loss; expert row offsets.
//   5. route_slots:     per tile, one warp walks its tokens in sequence order and
//                        gives each its slot = earlier tokens of the group with the
//                        same expert ("开源 AI 论文复现实验与代码解读 · 070",
//                        官方代码阅读路线: cumulative count along the sequence).
#include "common.cuh"
#include "kernels.h"

namespace smoe {

// ---------------------------------------------------------------- 1. router GEMM (CUDA cores, fp32)
constexpr int RL_BM = 64, RL_BN = 64, RL_BK = 16;

template <typename T>
__global__ void __launch_bounds__(256) router_logits_kernel(const T* __restrict__ x, const float* __restrict__ Wr,
                                                            const float* __restrict__ br, float* __restrict__ z,
                                                            int N, int d, int E) {
  __shared__ float xs[RL_BK][RL_BM + 4];
  __shared__ float ws[RL_BK][RL_BN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int n0 = blockIdx.y * RL_BM, e0 = blockIdx.x * RL_BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += RL_BK) {
    // 64 x 16 tiles, 4 elements per thread, stored k-major for broadcast reads
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = threadIdx.x + 256 * i;
      const int r = idx / RL_BK, k = idx % RL_BK;
      const int n = n0 + r, e = e0 + r, kk = k0 + k;
      xs[k][r] = (n < N && kk < d) ? ld_f32(x + (size_t)n * d + kk) : 0.f;
      ws[k][r] = (e < E && kk < d) ? Wr[(size_t)e * d + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < RL_BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = n0 + ty + 16 * i;
    if (n >= N) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx + 16 * j;
      if (e < E) z[(size_t)n * E + e] = acc[i][j] + (br ? br[e] : 0.f);
    }
  }
}

// ---------------------------------------------------------------- 2. softmax / top-1 per tile
// grid (nT, G), 256 threads.  Dynamic smem: hist[E] ints.
__global__ void __launch_bounds__(256) route_softmax_kernel(
    const float* __restrict__ z, int T, int E, int nT, int32_t* __restrict__ expert, float* __restrict__ gate,
    int32_t* __restrict__ tile_hist, float* __restrict__ tile_P, float* __restrict__ probs) {
  extern __shared__ int32_t hist[];
  __shared__ float m_s[ROUTE_TILE], s_s[ROUTE_TILE];
  const int g = blockIdx.y, tile = blockIdx.x;
  const int t0 = tile * ROUTE_TILE;
  const int len = min(ROUTE_TILE, T - t0);
  const size_t tok0 = (size_t)g * T + t0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
  for (int i = warp; i < len; i += nwarps) {
    const float* zr = z + (tok0 + i) * E;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {
      const float v = zr[e];
      if (v > best) { best = v; bi = e; }   // strict: first (lowest) index among equals
    }
    warp_argmax(best, bi);
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += expf(zr[e] - best);
    s = warp_sum(s);
    if (lane == 0) {
      m_s[i] = best;
      s_s[i] = s;
      expert[tok0 + i] = bi;
      gate[tok0 + i] = 1.0f / s;   // exp(z_top - max) / s with z_top = max
      atomicAdd(&hist[bi], 1);
    }
  }
  __syncthreads();

  // Column pass: probability sums per expert over the tile (fixed token order).
  const size_t tbase = ((size_t)g * nT + tile) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
    for (int i = 0; i < len; ++i) {
      const float p = expf(z[(tok0 + i) * E + e] - m_s[i]) / s_s[i];
      acc += p;
      if (probs) probs[(tok0 + i) * E + e] = p;
    }
    tile_P[tbase + e] = acc;
    tile_hist[tbase + e] = hist[e];
  }
}

// ---------------------------------------------------------------- 3. per (group, expert) scan over tiles
__global__ void route_scan_kernel(const int32_t* __restrict__ tile_hist, const float* __restrict__ tile_P,
                                  int32_t* __restrict__ tile_base, int32_t* __restrict__ raw,
                                  int32_t* __restrict__ accepted, float* __restrict__ P, int T, int E, int nT,
                                  int C) {
  const int g = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  int base = 0;
  float psum = 0.f;
  for (int j = 0; j < nT; ++j) {
    const size_t i = ((size_t)g * nT + j) * E + e;
    tile_base[i] = base;
    base += tile_hist[i];
    psum += tile_P[i];
  }
  raw[(size_t)g * E + e] = base;
  accepted[(size_t)g * E + e] = min(base, C);
  P[(size_t)g * E + e] = T > 0 ? psum / (float)T : 0.f;
}

// ---------------------------------------------------------------- 4. finalize (one CTA)
__global__ void __launch_bounds__(1024) route_finalize_kernel(
    const int32_t* __restrict__ raw, const int32_t* __restrict__ accepted, const float* __restrict__ P, int G,
    int T, int E, float alpha, float* __restrict__ balance, float* __restrict__ aux_g, float* __restrict__ aux,
    int32_t* __restrict__ group_off, int32_t* __restrict__ expert_rows) {
  __shared__ float red[1024];
  float total = 0.f;
  for (int g = 0; g < G; ++g) {
    float part = 0.f;
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      part += (float)raw[(size_t)g * E + e] * P[(size_t)g * E + e];
    red[threadIdx.x] = part;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      // E * sum_e f_e P_e with f_e = raw_e / T
      const float b = T > 0 ? (float)E * (red[0] / (float)T) : 0.f;
      balance[g] = b;
      aux_g[g] = alpha * b;
      total += alpha * b;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) aux[0] = G > 0 ? total / (float)G : 0.f;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int g = 0; g < G; ++g) {
      group_off[(size_t)g * E + e] = run;
      run += accepted[(size_t)g * E + e];
    }
    expert_rows[e] = run;
  }
}

// ---------------------------------------------------------------- 5. slots, one warp per tile
constexpr int SLOT_WARPS = 4;

__global__ void __launch_bounds__(SLOT_WARPS * 32) route_slots_kernel(
    const int32_t* __restrict__ expert, const int32_t* __restrict__ tile_base, const int32_t* __restrict__ group_off,
    int T, int E, int nT, int C, int R, int32_t* __restrict__ slot, uint8_t* __restrict__ keep,
    int32_t* __restrict__ row, int32_t* __restrict__ tok_of_row, bool debug, uint32_t* err) {
  extern __shared__ int32_t cnt_all[];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int g = blockIdx.y;
  const int tile = blockIdx.x * SLOT_WARPS + warp;
  if (tile >= nT) return;  // whole warp leaves; no block-wide barrier below
  int32_t* cnt = cnt_all + (size_t)warp * E;
  const size_t tb = ((size_t)g * nT + tile) * E;
  for (int e = lane; e < E; e += 32) cnt[e] = tile_base[tb + e];
  __syncwarp();
  const unsigned lt_mask = (1u << lane) - 1u;
  const int t_end = min(T, (tile + 1) * ROUTE_TILE);
  for (int t0 = tile * ROUTE_TILE; t0 < t_end; t0 += 32) {
    const int t = t0 + lane;
    const bool valid = t < t_end;
    const size_t tok = (size_t)g * T + t;
    int e = valid ? expert[tok] : -1 - lane;  // invalid lanes get keys of their own
    if (debug && valid && (e < 0 || e >= E)) { raise_error(err, ERR_BOUNDS); e = -1 - lane; }
    const bool live = e >= 0;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int base = live ? cnt[e] : 0;
    __syncwarp();
    if (live && lane == __ffs(same) - 1) cnt[e] = base + __popc(same);
    __syncwarp();
    if (valid) {
      const int s = base + __popc(same & lt_mask);
      const bool k = live && s < C;
      slot[tok] = s;
      keep[tok] = k ? 1 : 0;
      int r = -1;
      if (k) {
        r = group_off[(size_t)g * E + e] + s;
        if (debug && (r < 0 || r >= R)) { raise_error(err, ERR_BOUNDS); r = -1; }
        else tok_of_row[(size_t)e * R + r] = (int32_t)tok;
      }
      row[tok] = r;
    }
  }
}

// ---------------------------------------------------------------- launcher
int launch_route(const RouteArgs& a, cudaStream_t s) {
  const int N = a.G * a.T;
  const int nT = (a.T + ROUTE_TILE - 1) / ROUTE_TILE;
  int launches = 0;
  if (N > 0) {
    dim3 grid((a.E + RL_BN - 1) / RL_BN, (N + RL_BM - 1) / RL_BM);
    if (a.x_bf16)
      router_logits_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>((const __nv_bfloat16*)a.x, a.Wr, a.br, a.logits,
                                                               N, a.d, a.E);
    else
      router_logits_kernel<float><<<grid, 256, 0, s>>>((const float*)a.x, a.Wr, a.br, a.logits, N, a.d, a.E);
    ++launches;
    route_softmax_kernel<<<dim3(nT, a.G), 256, a.E * sizeof(int32_t), s>>>(
        a.logits, a.T, a.E, nT, a.expert, a.gate, a.tile_hist, a.tile_P, a.probs);
    ++launches;
  }
  route_scan_kernel<<<dim3((a.E + 255) / 256, a.G), 256, 0, s>>>(a.tile_hist, a.tile_P, a.tile_base, a.raw,
                                                                 a.accepted, a.P, a.T, a.E, nT, a.C);
  ++launches;
  route_finalize_kernel<<<1, 1024, 0, s>>>(a.raw, a.accepted, a.P, a.G, a.T, a.E, a.alpha, a.balance, a.aux_g,
                                           a.aux, a.group_off, a.expert_rows);
  ++launches;
  if (N > 0) {
    route_slots_kernel<<<dim3((nT + SLOT_WARPS - 1) / SLOT_WARPS, a.G), SLOT_WARPS * 32,
                         SLOT_WARPS * a.E * sizeof(int32_t), s>>>(a.expert, a.tile_base, a.group_off, a.T, a.E,
                                                                  nT, a.C, a.R, a.slot, a.keep, a.row,
                                                                  a.tok_of_row, a.debug, a.err);
    ++launches;
  }
  if (cudaGetLastError() != cudaSuccess) return -1;
  return launches;
}

}  // namespace smoe
