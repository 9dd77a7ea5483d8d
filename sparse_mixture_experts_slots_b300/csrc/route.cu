// Routing kernels of the top-1 Switch layer (sm_103a).
//
// Stages, following the pipeline of "042 · Switch Transformer：每个词只选一个专家",
// section 三 (float32 router -> one expert per token -> load statistics and aux
// loss -> capacity truncation):
//   1. router:   z = x W_r^T + b_r in float32 (x cast up; selective precision,
//                Switch Transformers card on ai-papers.xuzou.cn, 方法适配), softmax,
//                top-1 (ties -> lowest index), gate, and per 128-token tile the expert
//                histogram, the probability sums and each token's rank among the
//                tile's earlier tokens with the same expert.  bf16 activations use the
//                tensor-core kernel in route_tc.cu; float32 activations use the
//                CUDA-core kernels below (router_logits + route_softmax).
//   2. route_scan: per (group, expert) exclusive prefix of the tile histograms, raw
//                and accepted counts, mean probability P, expert row offsets; the last
//                block computes each group's balance E * sum f P, its aux loss and
//                the mean over groups.
//   3. slots:    slot = (tokens of the group's earlier tiles with the same expert)
//                + rank, i.e. the cumulative count along the sequence
//                ("开源 AI 论文复现实验与代码解读 · 070", 官方代码阅读路线);
//                keep = slot < C; row in the expert's block of the dispatched buffer.
#include "common.cuh"
#include "kernels.h"

namespace smoe {

// ---------------------------------------------------------------- 1. router GEMM (CUDA cores, fp32)
constexpr int RL_BM = 64, RL_BN = 64, RL_BK = 16;

template <typename T>
__global__ void __launch_bounds__(256) router_logits_kernel(const T* __restrict__ x, const float* __restrict__ Wr,
                                                            const float* __restrict__ br, float* __restrict__ z,
                                                            int N, int d, int E) {
  griddep_wait();
  griddep_launch_dependents();
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

// ---------------------------------------------------------------- 2. softmax / top-1 per tile (float32 path)
// grid (nT, G), 256 threads.  Dynamic smem: hist[E] ints.  Writes the in-tile rank to rank[].
__global__ void __launch_bounds__(256) route_softmax_kernel(
    const float* __restrict__ z, int T, int E, int nT, int32_t* __restrict__ expert, float* __restrict__ gate,
    int32_t* __restrict__ rank, int32_t* __restrict__ tile_hist, float* __restrict__ tile_P,
    float* __restrict__ tile_Z, float* __restrict__ probs, uint32_t* err) {
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ int32_t hist[];
  __shared__ float m_s[ROUTE_TILE], s_s[ROUTE_TILE], zz_s[ROUTE_TILE];
  __shared__ int a_s[ROUTE_TILE];
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
    if (bi < 0 || bi >= E) {  // non-finite logits only
      if (lane == 0) raise_error(err, ERR_BOUNDS);
      bi = 0;
    }
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += expf(zr[e] - best);
    s = warp_sum(s);
    if (lane == 0) {
      m_s[i] = best;
      s_s[i] = s;
      a_s[i] = bi;
      const float lse = best + logf(s);  // log sum_e exp z_e, for the router z-loss
      zz_s[i] = lse * lse;
      expert[tok0 + i] = bi;
      gate[tok0 + i] = 1.0f / s;   // exp(z_top - max) / s with z_top = max
      atomicAdd(&hist[bi], 1);
    }
  }
  __syncthreads();

  // the tile's sum of (log sum exp z)^2, in a fixed order
  if (warp == 0) {
    float zs = 0.f;
    for (int i = lane; i < len; i += 32) zs += zz_s[i];
    zs = warp_sum(zs);
    if (lane == 0) tile_Z[(size_t)g * nT + tile] = zs;
  }

  // rank among the tile's earlier tokens with the same expert
  for (int i = threadIdx.x; i < len; i += blockDim.x) {
    int r = 0;
    for (int j = 0; j < i; ++j) r += a_s[j] == a_s[i];
    rank[tok0 + i] = r;
  }

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

// ---------------------------------------------------------------- 2b. top-2 per tile (from float32 logits)
// grid (nT, G), 512 threads; dynamic smem: hist[E], hist2[E] ints, then the column pass's
// partial sums [ceil(512 / E)][E] floats.  Per token: the two
// highest logits (ties to the lower index), their weights = softmax over the two, the
// full softmax's column sums (P), (log sum exp z)^2, and the in-tile ranks of both
// choices among the tile's first / second choices (into rank[] / rank2[]).
__device__ __forceinline__ bool top_before(float v, int i, float w, int j) {
  return v > w || (v == w && i < j);  // (v, i) ranks before (w, j)
}

constexpr int TOP2_THREADS = 512;
constexpr float ROUTE_LOG2E = 1.4426950408889634f;

__global__ void __launch_bounds__(TOP2_THREADS) route_top2_kernel(
    const float* __restrict__ z, int T, int E, int nT, int32_t* __restrict__ expert, int32_t* __restrict__ expert2,
    float* __restrict__ gate, float* __restrict__ gate2, int32_t* __restrict__ rank, int32_t* __restrict__ rank2,
    int32_t* __restrict__ tile_hist, int32_t* __restrict__ tile_hist2, float* __restrict__ tile_P,
    float* __restrict__ tile_Z, float* __restrict__ probs, uint32_t* err, int staged) {
  griddep_wait();
  griddep_launch_dependents();
  // [2E] ints: first choices, then second choices; [nch E] floats: column partials; with
  // `staged`, the tile's logits [ROUTE_TILE][E] (each token's row becomes its probabilities)
  extern __shared__ __align__(16) int32_t hist[];
  int32_t* hist2 = hist + E;
  __shared__ float m_s[ROUTE_TILE], r_s[ROUTE_TILE], zz_s[ROUTE_TILE];  // max, 1 / sum exp, lse^2
  __shared__ int a_s[ROUTE_TILE], a2_s[ROUTE_TILE];
  __shared__ uint64_t stage_bar;
  __shared__ int stage_ok;
  const int g = blockIdx.y, tile = blockIdx.x;
  const int t0 = tile * ROUTE_TILE;
  const int len = min(ROUTE_TILE, T - t0);
  const size_t tok0 = (size_t)g * T + t0;
  for (int e = threadIdx.x; e < 2 * E; e += blockDim.x) hist[e] = 0;
  const int nch = E >= (int)blockDim.x ? 1 : (int)blockDim.x / E;
  float* zt = reinterpret_cast<float*>(hist + 2 * E) + (size_t)nch * E;  // staged logits
  // The tile's rows are contiguous: one bulk copy into shared memory when E allows 16-byte
  // alignment (E % 4 == 0; at most 200 KB, under an mbarrier's transaction limit).
  const bool bulk = staged && (E & 3) == 0;
  if (bulk && threadIdx.x == 0) {
    mbar_init(&stage_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (bulk) {
    if (threadIdx.x == 0) {
      const uint32_t bytes = (uint32_t)((size_t)len * E * sizeof(float));
      mbar_arrive_expect_tx(&stage_bar, bytes);
      bulk_load(zt, z + tok0 * E, bytes, &stage_bar);
      stage_ok = mbar_wait(&stage_bar, 0) ? 1 : 0;
    }
  } else if (staged) {
    for (int k = threadIdx.x; k < len * E; k += blockDim.x) zt[k] = z[tok0 * E + k];
  }
  __syncthreads();
  if (bulk && !stage_ok) {  // the copy never landed (bounded wait): report, leave the tile
    if (threadIdx.x == 0) raise_error(err, ERR_TIMEOUT);
    return;
  }

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nwarps = blockDim.x / 32;
  for (int i = warp; i < len; i += nwarps) {
    const float* zr = staged ? zt + (size_t)i * E : z + (tok0 + i) * E;
    float m1 = -INFINITY, m2 = -INFINITY;
    int i1 = 0x7fffffff, i2 = 0x7fffffff;
    for (int e = lane; e < E; e += 32) {  // increasing e: strict > keeps the lower index
      const float v = zr[e];
      if (v > m1) {
        m2 = m1; i2 = i1; m1 = v; i1 = e;
      } else if (v > m2) {
        m2 = v; i2 = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {  // merge the lanes' pairs (indices are distinct)
      const float p1 = __shfl_xor_sync(0xffffffffu, m1, o), p2 = __shfl_xor_sync(0xffffffffu, m2, o);
      const int j1 = __shfl_xor_sync(0xffffffffu, i1, o), j2 = __shfl_xor_sync(0xffffffffu, i2, o);
      if (top_before(p1, j1, m1, i1)) {
        if (!top_before(m1, i1, p2, j2)) { m2 = p2; i2 = j2; } else { m2 = m1; i2 = i1; }
        m1 = p1; i1 = j1;
      } else if (top_before(p1, j1, m2, i2)) {
        m2 = p1; i2 = j1;
      }
    }
    if (i1 < 0 || i1 >= E || i2 < 0 || i2 >= E || i1 == i2) {  // non-finite logits only
      if (lane == 0) raise_error(err, ERR_BOUNDS);
      i1 = 0;
      i2 = 1;
      m1 = zr[0];
      m2 = zr[1];
    }
    // exp(z - m1) as 2^(z log2 e - m1 log2 e) on the special-function unit
    const float m1s = m1 * ROUTE_LOG2E;
    float s = 0.f;
    for (int e = lane; e < E; e += 32) s += ex2_approx(fmaf(zr[e], ROUTE_LOG2E, -m1s));
    s = warp_sum(s);
    const float rs = 1.0f / s;
    if (staged) {  // the row's probabilities in place (each lane rewrites only what it read)
      float* pr = zt + (size_t)i * E;
      for (int e = lane; e < E; e += 32) {
        const float pv = ex2_approx(fmaf(pr[e], ROUTE_LOG2E, -m1s)) * rs;
        pr[e] = pv;
        if (probs) probs[(tok0 + i) * E + e] = pv;
      }
    }
    if (lane == 0) {
      m_s[i] = m1;
      r_s[i] = rs;
      a_s[i] = i1;
      a2_s[i] = i2;
      const float u = ex2_approx((m2 - m1) * ROUTE_LOG2E);  // the pair's softmax: 1 / (1 + u), u / (1 + u)
      expert[tok0 + i] = i1;
      expert2[tok0 + i] = i2;
      gate[tok0 + i] = 1.0f / (1.0f + u);
      gate2[tok0 + i] = u / (1.0f + u);
      const float lse = m1 + logf(s);
      zz_s[i] = lse * lse;
      atomicAdd(&hist[i1], 1);
      atomicAdd(&hist2[i2], 1);
    }
  }
  __syncthreads();

  if (warp == 0) {  // the tile's sum of (log sum exp z)^2, in a fixed order
    float zs = 0.f;
    for (int i = lane; i < len; i += 32) zs += zz_s[i];
    zs = warp_sum(zs);
    if (lane == 0) tile_Z[(size_t)g * nT + tile] = zs;
  }
  for (int i = threadIdx.x; i < len; i += blockDim.x) {
    int r = 0, r2 = 0;
    for (int j = 0; j < i; ++j) {
      r += a_s[j] == a_s[i];
      r2 += a2_s[j] == a2_s[i];
    }
    rank[tok0 + i] = r;
    rank2[tok0 + i] = r2;
  }
  // Column pass: (expert, token chunk) per thread, chunk sums combined in a fixed order.
  const size_t tbase = ((size_t)g * nT + tile) * E;
  float* part = reinterpret_cast<float*>(hist + 2 * E);
  const int clen = (len + nch - 1) / nch;
  for (int k = threadIdx.x; k < E * nch; k += blockDim.x) {
    const int e = k % E, c = k / E;
    float acc = 0.f;
    const int i1 = min(len, (c + 1) * clen);
    if (staged) {
      for (int i = c * clen; i < i1; ++i) acc += zt[(size_t)i * E + e];
    } else {
      for (int i = c * clen; i < i1; ++i) {
        const float p = ex2_approx(fmaf(z[(tok0 + i) * E + e], ROUTE_LOG2E, -m_s[i] * ROUTE_LOG2E)) * r_s[i];
        acc += p;
        if (probs) probs[(tok0 + i) * E + e] = p;
      }
    }
    part[c * E + e] = acc;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
    for (int c = 0; c < nch; ++c) acc += part[c * E + e];
    tile_P[tbase + e] = acc;
    tile_hist[tbase + e] = hist[e];
    tile_hist2[tbase + e] = hist2[e];
  }
}

// ---------------------------------------------------------------- 3. cross-tile scan + finalize
// One block per (32 experts, routing group), lane <-> expert; the warps split the group's
// tiles.  Each block writes its group's tile prefixes, raw / accepted counts and P; the last
// block to finish (atomic ticket) adds the groups' row counts in group order (group row
// offsets, expert block rows) and the per-block balance partials in a fixed order.  When the
// router z-loss is asked for, one more block reduces the tiles' sums of (log sum exp z)^2 per
// group, alongside the scan (nothing later in the layer waits for it).
constexpr int SCAN_WARPS = 16;

__global__ void __launch_bounds__(SCAN_WARPS * 32) route_scan_kernel(
    const int32_t* __restrict__ tile_hist, const float* __restrict__ tile_P, const float* __restrict__ tile_Z,
    const int32_t* __restrict__ tile_hist2, int G, int T, int E, int nT, int C, float alpha,
    int32_t* __restrict__ tile_base, int32_t* __restrict__ tile_base2, int32_t* __restrict__ raw,
    int32_t* __restrict__ accepted, int32_t* __restrict__ raw2, int32_t* __restrict__ accepted2,
    float* __restrict__ P, int32_t* __restrict__ group_off,
    int32_t* __restrict__ expert_rows, float* __restrict__ balance, float* __restrict__ aux_g,
    float* __restrict__ aux, float* __restrict__ z_g, float* __restrict__ z, float* __restrict__ partial,
    uint32_t* __restrict__ counter) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int sh_h[SCAN_WARPS][32], sh_h2[SCAN_WARPS][32];
  __shared__ float sh_p[SCAN_WARPS][32];
  __shared__ double sh_z[SCAN_WARPS];
  __shared__ int is_last;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nblk = route_scan_blocks(E);
  if ((int)blockIdx.x >= nblk) {  // router z-loss: a warp per group, then the mean over groups
    if (blockIdx.y != 0) return;
    double wsum = 0.0;
    for (int g = warp; g < G; g += SCAN_WARPS) {
      double zs = 0.0;
      for (int j = lane; j < nT; j += 32) zs += (double)tile_Z[(size_t)g * nT + j];
      zs = warp_sum_d(zs);
      const float zg = T > 0 ? (float)(zs / (double)T) : 0.f;
      if (lane == 0 && z_g) z_g[g] = zg;
      wsum += (double)zg;
    }
    if (lane == 0) sh_z[warp] = wsum;
    __syncthreads();
    if (threadIdx.x == 0 && z) {
      double zt = 0.0;
      for (int w = 0; w < SCAN_WARPS; ++w) zt += sh_z[w];
      z[0] = G > 0 ? (float)(zt / (double)G) : 0.f;
    }
    return;
  }
  const int g = blockIdx.y;
  const int e = blockIdx.x * 32 + lane;
  const bool ev = e < E;
  const int chunk = (nT + SCAN_WARPS - 1) / SCAN_WARPS;
  const int j0 = min(nT, warp * chunk), j1 = min(nT, j0 + chunk);
  {
    int hs = 0, hs2 = 0;
    float ps = 0.f;
    if (ev)
      for (int j = j0; j < j1; ++j) {
        const size_t idx = ((size_t)g * nT + j) * E + e;
        hs += tile_hist[idx];
        ps += tile_P[idx];
        if (tile_hist2) hs2 += tile_hist2[idx];  // top-2: second choices, counted the same way
      }
    sh_h[warp][lane] = hs;
    sh_h2[warp][lane] = hs2;
    sh_p[warp][lane] = ps;
    __syncthreads();
    int base = 0, base2 = 0;
    for (int w = 0; w < warp; ++w) {
      base += sh_h[w][lane];
      base2 += sh_h2[w][lane];
    }
    if (ev)
      for (int j = j0; j < j1; ++j) {
        const size_t idx = ((size_t)g * nT + j) * E + e;
        tile_base[idx] = base;
        base += tile_hist[idx];
        if (tile_hist2) {
          tile_base2[idx] = base2;
          base2 += tile_hist2[idx];
        }
      }
    if (warp == 0) {
      int tot = 0, tot2 = 0;
      float psum = 0.f;
      for (int w = 0; w < SCAN_WARPS; ++w) {
        tot += sh_h[w][lane];
        tot2 += sh_h2[w][lane];
        psum += sh_p[w][lane];
      }
      float contrib = 0.f;
      if (ev) {
        const size_t ge = (size_t)g * E + e;
        const int acc = min(tot, C);
        const float Pv = T > 0 ? psum / (float)T : 0.f;
        raw[ge] = tot;
        accepted[ge] = acc;
        P[ge] = Pv;
        if (tile_hist2) {  // second choices fill what the kept first choices leave
          raw2[ge] = tot2;
          accepted2[ge] = min(tot2, max(C - acc, 0));
        }
        contrib = (float)tot * Pv;
      }
      contrib = warp_sum(contrib);
      if (lane == 0) partial[(size_t)g * nblk + blockIdx.x] = contrib;
    }
  }

  // The last block to finish: group row offsets and expert rows (groups in order), then the
  // per-block partials (fixed order) per group.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(counter, 1u) == (unsigned)(nblk * G) - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int ee = threadIdx.x; ee < E; ee += blockDim.x) {
    int rows_run = 0;
    for (int gg = 0; gg < G; ++gg) {
      const size_t ge = (size_t)gg * E + ee;
      group_off[ge] = rows_run;
      rows_run += __ldcg(&accepted[ge]);
      if (tile_hist2) rows_run += __ldcg(&accepted2[ge]);
    }
    expert_rows[ee] = rows_run;
  }
  for (int gg = threadIdx.x; gg < G; gg += blockDim.x) {
    float sum = 0.f;
    for (int b = 0; b < nblk; ++b) sum += __ldcg(&partial[(size_t)gg * nblk + b]);
    // E * sum_e f_e P_e with f_e = raw_e / T
    const float bal = T > 0 ? (float)E * (sum / (float)T) : 0.f;
    balance[gg] = bal;
    aux_g[gg] = alpha * bal;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float total = 0.f;
    for (int gg = 0; gg < G; ++gg) total += aux_g[gg];
    aux[0] = G > 0 ? total / (float)G : 0.f;
    *counter = 0u;
  }
}

// ---------------------------------------------------------------- 4. slots, one thread per token
__global__ void __launch_bounds__(256) route_slots_kernel(
    const int32_t* __restrict__ expert, const int32_t* __restrict__ tile_base, const int32_t* __restrict__ group_off,
    long long N, int T, int E, int nT, int C, int R, int32_t* __restrict__ slot, uint8_t* __restrict__ keep,
    int32_t* __restrict__ row, int32_t* __restrict__ tok_of_row, bool debug, uint32_t* err) {
  griddep_wait();
  griddep_launch_dependents();
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (t >= N) return;
  const int g = (int)(t / T);
  const int ti = (int)(t - (long long)g * T);
  const int e = expert[t];
  if (e < 0 || e >= E) {  // the router never writes one; keep every access in bounds regardless
    raise_error(err, ERR_BOUNDS);
    slot[t] = 0;
    keep[t] = 0;
    row[t] = -1;
    return;
  }
  const int s = tile_base[((size_t)g * nT + ti / ROUTE_TILE) * E + e] + slot[t];  // slot[] holds the rank
  const bool k = s < C;
  slot[t] = s;
  keep[t] = k ? 1 : 0;
  int r = -1;
  if (k) {
    r = group_off[(size_t)g * E + e] + s;
    if (r < 0 || r >= R) {
      if (debug) raise_error(err, ERR_BOUNDS);
      r = -1;
      keep[t] = 0;
    } else {
      tok_of_row[(size_t)e * R + r] = (int32_t)t;
    }
  }
  row[t] = r;
}

// top-2: slots of both choices.  A first choice is numbered among the group's first
// choices of its expert; a second choice after that expert's kept first choices, among
// the group's second choices.  Rows: group_off + slot (kept first choices, then kept
// second choices, in each expert's block of the group).
__global__ void __launch_bounds__(256) route_slots_top2_kernel(
    const int32_t* __restrict__ expert, const int32_t* __restrict__ expert2, const int32_t* __restrict__ tile_base,
    const int32_t* __restrict__ tile_base2, const int32_t* __restrict__ group_off,
    const int32_t* __restrict__ accepted, long long N, int T, int E, int nT, int C, int R,
    int32_t* __restrict__ slot, int32_t* __restrict__ slot2, uint8_t* __restrict__ keep, uint8_t* __restrict__ keep2,
    int32_t* __restrict__ row, int32_t* __restrict__ row2, int32_t* __restrict__ tok_of_row, bool debug,
    uint32_t* err) {
  griddep_wait();
  griddep_launch_dependents();
  const long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (t >= N) return;
  const int g = (int)(t / T);
  const int ti = (int)(t - (long long)g * T);
  const size_t tb = ((size_t)g * nT + ti / ROUTE_TILE) * E;
  for (int k = 0; k < 2; ++k) {
    const int e = k ? expert2[t] : expert[t];
    int32_t* sl = k ? slot2 : slot;
    uint8_t* kp = k ? keep2 : keep;
    int32_t* rw = k ? row2 : row;
    if (e < 0 || e >= E) {  // the router never writes one; keep every access in bounds regardless
      raise_error(err, ERR_BOUNDS);
      sl[t] = 0;
      kp[t] = 0;
      rw[t] = -1;
      continue;
    }
    const int s = k ? accepted[(size_t)g * E + e] + tile_base2[tb + e] + sl[t] : tile_base[tb + e] + sl[t];
    const bool kept = s < C;
    int r = -1;
    if (kept) {
      r = group_off[(size_t)g * E + e] + s;
      if (r < 0 || r >= R) {
        if (debug) raise_error(err, ERR_BOUNDS);
        r = -1;
      } else {
        tok_of_row[(size_t)e * R + r] = (int32_t)t;
      }
    }
    sl[t] = s;
    kp[t] = r >= 0 ? 1 : 0;
    rw[t] = r;
  }
}

// ---------------------------------------------------------------- launcher
int launch_route(const RouteArgs& a, cudaStream_t s) {
  const long long N = (long long)a.G * a.T;
  const int nT = (a.T + ROUTE_TILE - 1) / ROUTE_TILE;
  int launches = 0;
  if (N > 0 && a.top2 && a.x_bf16 && router_tc_top2_fused(a.E, a.d)) {
    // top-2 in the tensor-core router's own pass (no float32 logits round trip)
    const int n = launch_router_tc(a, a.slot, s);
    if (n < 0) return -1;
    launches += n;
  } else if (N > 0 && a.top2) {
    // top-2: float32 logits from the router (tensor cores for bf16 x: its own top-1
    // outputs are overwritten below), then the per-tile top-2 pass
    if (a.x_bf16) {
      RouteArgs b = a;
      b.logits_out = a.logits;
      b.top2 = false;
      const int n = launch_router_tc(b, a.slot, s);
      if (n < 0) return -1;
      launches += n;
    } else {
      dim3 grid((a.E + RL_BN - 1) / RL_BN, (unsigned)((N + RL_BM - 1) / RL_BM));
      if (launch_k(router_logits_kernel<float>, grid, dim3(256), 0, s, false, 1, (const float*)a.x, a.Wr, a.br,
                   a.logits, (int)N, a.d, a.E) != cudaSuccess)
        return -1;
      ++launches;
    }
    const int nch = a.E >= TOP2_THREADS ? 1 : TOP2_THREADS / a.E;
    // the tile's logits staged in shared memory when they fit (E up to about 390)
    const size_t base_smem = 2 * a.E * sizeof(int32_t) + (size_t)nch * a.E * sizeof(float);
    const size_t stage_smem = (size_t)ROUTE_TILE * a.E * sizeof(float);
    const int staged = base_smem + stage_smem <= 200 * 1024 ? 1 : 0;
    const size_t smem = base_smem + (staged ? stage_smem : 0);
    // the attribute is the bound every call stays under (one value whatever the shape, so
    // calls from several host threads never lower it under one another's launch)
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(route_top2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
      return -1;
    if (launch_k(route_top2_kernel, dim3(nT, a.G), dim3(TOP2_THREADS), smem, s, true, 1, (const float*)a.logits, a.T,
                 a.E, nT, a.expert, a.expert2, a.gate, a.gate2, a.slot, a.slot2, a.tile_hist, a.tile_hist2, a.tile_P,
                 a.tile_Z, a.probs, a.err, staged) != cudaSuccess)
      return -1;
    ++launches;
  } else if (N > 0) {
    if (a.x_bf16) {
      const int n = launch_router_tc(a, a.slot, s);
      if (n < 0) return -1;
      launches += n;
    } else {
      dim3 grid((a.E + RL_BN - 1) / RL_BN, (unsigned)((N + RL_BM - 1) / RL_BM));
      if (launch_k(router_logits_kernel<float>, grid, dim3(256), 0, s, false, 1, (const float*)a.x, a.Wr, a.br,
                   a.logits, (int)N, a.d, a.E) != cudaSuccess ||
          launch_k(route_softmax_kernel, dim3(nT, a.G), dim3(256), a.E * sizeof(int32_t), s, true, 1, a.logits, a.T,
                   a.E, nT, a.expert, a.gate, a.slot, a.tile_hist, a.tile_P, a.tile_Z, a.probs, a.err) != cudaSuccess)
        return -1;
      launches += 2;
    }
  }
  // The scan follows the router kernel of this call (programmatic launch); with no
  // tokens it is the first kernel of the call.
  const int scan_grid = route_scan_blocks(a.E) + ((a.z_g || a.z) ? 1 : 0);
  if (a.G > 65535) return -1;
  if (launch_k(route_scan_kernel, dim3(scan_grid, a.G), dim3(SCAN_WARPS * 32), 0, s, N > 0, 1, a.tile_hist,
               a.tile_P, (const float*)a.tile_Z, a.top2 ? (const int32_t*)a.tile_hist2 : nullptr, a.G, a.T, a.E, nT,
               a.C, a.alpha, a.tile_base, a.top2 ? a.tile_base2 : nullptr, a.raw, a.accepted,
               a.top2 ? a.raw2 : nullptr, a.top2 ? a.accepted2 : nullptr, a.P, a.group_off, a.expert_rows,
               a.balance, a.aux_g, a.aux, a.z_g, a.z, a.scan_partial, a.scan_counter) != cudaSuccess)
    return -1;
  ++launches;
  if (N > 0 && a.top2) {
    if (launch_k(route_slots_top2_kernel, dim3((unsigned)((N + 255) / 256)), dim3(256), 0, s, true, 1, a.expert,
                 a.expert2, a.tile_base, a.tile_base2, a.group_off, a.accepted, N, a.T, a.E, nT, a.C, a.R, a.slot,
                 a.slot2, a.keep, a.keep2, a.row, a.row2, a.tok_of_row, a.debug, a.err) != cudaSuccess)
      return -1;
    ++launches;
  } else if (N > 0 && a.slots) {
    if (launch_k(route_slots_kernel, dim3((unsigned)((N + 255) / 256)), dim3(256), 0, s, true, 1, a.expert,
                 a.tile_base, a.group_off, N, a.T, a.E, nT, a.C, a.R, a.slot, a.keep, a.row, a.tok_of_row, a.debug,
                 a.err) != cudaSuccess)
      return -1;
    ++launches;
  }
  if (cudaGetLastError() != cudaSuccess) return -1;
  return launches;
}

}  // namespace smoe
