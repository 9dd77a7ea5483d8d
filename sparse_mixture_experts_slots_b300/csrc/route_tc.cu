// Router of the top-1 Switch layer on 5th-generation tensor cores (tcgen05, sm_103a).
//
// The router runs in float32 (selective precision: Switch Transformers card on
// ai-papers.xuzou.cn, 方法适配; "042 · Switch Transformer：每个词只选一个专家",
// section 一, p(x) = softmax(W_r x)).  The activations are bfloat16, so every x_k
// is exact in bfloat16; W_r is float32 and is split into three bfloat16 pieces
// hi + mid + lo whose sum equals w to within 2^-24 |w| (each piece holds the
// next 8 bits of the significand).  Then
//     z = x . hi + x . (mid + lo)
// with every bf16 x bf16 product exact and accumulated in float32 by the tensor
// cores: two TMEM accumulators (hi and the correction) so the small terms do not
// share an accumulator with the large ones; they are added in the epilogue.
//
// One CTA (or a cluster of Q CTAs, each with EC experts) takes a tile of 128
// tokens of one routing group:
//   warp 0, one lane : TMA producer (x tiles in one ring, W_r pieces in another)
//   warp 1, one lane : MMA issuer (M = 128 tokens, N = EC experts, K = 16 per op)
//   4 warps          : epilogue; thread i owns token i (TMEM lane i):
//     pass 1  logits z (+ bias), local max / argmax (ties -> lowest index), local sum
//     exchange of (max, sum, argmax) between the Q CTAs through distributed shared memory
//     pass 2  p = exp(z - max) / sum; column sums over the tile's tokens (warp
//             reduce-scatter), expert histogram of the tile, rank of each token
//             among the tile's earlier tokens with the same expert.
// Outputs per token: expert (raw choice), gate = p_{expert}, rank in tile; per
// (group, tile, expert): token count and probability sum.  The cross-tile scan
// that turns ranks into slots runs in route.cu.
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int RT_BM = ROUTE_TILE;  // 128 tokens per tile
constexpr int RT_BK = 64;          // 64 bf16 = one 128-byte swizzle row

// ---------------------------------------------------------------- W_r -> hi, mid, lo
__global__ void router_split_kernel(const float* __restrict__ Wr, __nv_bfloat16* __restrict__ ws, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float w = Wr[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);  // exact: fits in the 24-bit significand
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);  // exact
    ws[i] = hi;
    ws[n + i] = mid;
    ws[2 * n + i] = __float2bfloat16_rn(r2);
  }
}

// ---------------------------------------------------------------- shared memory layout
template <int EC>
struct RtCfg {
  static constexpr int XS = EC >= 128 ? 2 : 3;  // x-tile ring depth
  static constexpr int WS = EC >= 128 ? 4 : 6;  // W-piece ring depth
  static constexpr int X_BYTES = RT_BM * RT_BK * 2;
  static constexpr int W_BYTES = EC * RT_BK * 2;
  static constexpr int RING_BYTES = XS * X_BYTES + WS * W_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * EC < 32 ? 32 : 2 * EC;  // hi + correction accumulators
  static_assert(EC % 16 == 0 && EC >= 16 && EC <= 256, "tcgen05 M=128 takes N = 16..256 in steps of 16");
  static_assert((EC & (EC - 1)) == 0, "EC is a power of two (TMEM allocation)");
  static_assert(X_BYTES % 1024 == 0 && W_BYTES % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

template <int EC>
struct RtShared {
  uint64_t xfull[RtCfg<EC>::XS], xempty[RtCfg<EC>::XS];
  uint64_t wfull[RtCfg<EC>::WS], wempty[RtCfg<EC>::WS];
  uint64_t accb;
  uint32_t tmem_slot;
  volatile int abort_flag;
  float m[RT_BM];     // local (this CTA's experts) max logit per token
  float s[RT_BM];     // local sum of exp(z - m)
  int a[RT_BM];       // local argmax
  int texp[RT_BM];    // final expert per token (-1 past the group's end)
  float colsum[4][EC];
  int hist[EC];
  float bias[EC];
};

template <int EC>
constexpr int rt_smem_bytes() {
  return RtCfg<EC>::RING_BYTES + (int)sizeof(RtShared<EC>) + 1024;
}

// Sum of v over the 32 lanes for 16 columns at once (reduce-scatter).  On return,
// lane L holds the warp's total of column (L >> 1) & 15 (lanes L and L^1 agree).
__device__ __forceinline__ float warp_colsum16(const float (&p)[16], int lane) {
  float v8[8], v4[4], v2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float send = b4 ? p[j] : p[j + 8];
    const float keep = b4 ? p[j + 8] : p[j];
    v8[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = b3 ? v8[j] : v8[j + 4];
    const float keep = b3 ? v8[j + 4] : v8[j];
    v4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = b2 ? v4[j] : v4[j + 2];
    const float keep = b2 ? v4[j + 2] : v4[j];
    v2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const float send = b1 ? v2[0] : v2[1];
  const float keep = b1 ? v2[1] : v2[0];
  const float v1 = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  return v1 + __shfl_xor_sync(0xffffffffu, v1, 1);
}

// ---------------------------------------------------------------- the router kernel
// grid (Q * nT, G); clusters of Q CTAs along x when Q > 1.
template <int EC>
__global__ void __launch_bounds__(128, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const float* __restrict__ br, int T, int E, int d, int nT, int Q,
                     int32_t* __restrict__ expert, float* __restrict__ gate, int32_t* __restrict__ rank,
                     int32_t* __restrict__ tile_hist, float* __restrict__ tile_P, float* __restrict__ logits,
                     float* __restrict__ probs, uint32_t* err) {
  using Cf = RtCfg<EC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = smem;
  uint8_t* sW = smem + Cf::XS * Cf::X_BYTES;
  RtShared<EC>& sh = *reinterpret_cast<RtShared<EC>*>(smem + Cf::RING_BYTES);

  const int q = Q > 1 ? (int)cluster_ctarank() : 0;
  const int tile = blockIdx.x / Q;
  const int g = blockIdx.y;
  const int e0 = q * EC;
  const int t0 = tile * RT_BM;
  const long long tok0 = (long long)g * T + t0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int KB = (d + RT_BK - 1) / RT_BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cf::XS; ++i) {
      mbar_init(&sh.xfull[i], 1);
      mbar_init(&sh.xempty[i], 1);
    }
    for (int i = 0; i < Cf::WS; ++i) {
      mbar_init(&sh.wfull[i], 1);
      mbar_init(&sh.wempty[i], 1);
    }
    mbar_init(&sh.accb, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  for (int c = threadIdx.x; c < EC; c += blockDim.x) {
    const int e = e0 + c;
    sh.bias[c] = (br && e < E) ? br[e] : 0.f;
    sh.hist[c] = 0;
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_slot, Cf::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int xi = 0, wi = 0;  // loads issued into each ring
    bool ok = true;
    for (int kb = 0; kb < KB && ok; ++kb) {
      const int xs = kb % Cf::XS;
      if (kb >= Cf::XS && !mbar_wait(&sh.xempty[xs], ((kb / Cf::XS) - 1) & 1)) { ok = false; break; }
      if (sh.abort_flag) { ok = false; break; }
      mbar_arrive_expect_tx(&sh.xfull[xs], Cf::X_BYTES);
      tma_load_2d(sX + xs * Cf::X_BYTES, &tmX, &sh.xfull[xs], kb * RT_BK, (int)tok0);
      xi = kb + 1;
      for (int s = 0; s < 3; ++s) {
        const int j = kb * 3 + s, ws = j % Cf::WS;
        if (j >= Cf::WS && !mbar_wait(&sh.wempty[ws], ((j / Cf::WS) - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&sh.wfull[ws], Cf::W_BYTES);
        tma_load_2d(sW + ws * Cf::W_BYTES, &tmW, &sh.wfull[ws], kb * RT_BK, s * E + e0);
        wi = j + 1;
      }
    }
    if (!ok) {
      raise_error(err, ERR_TIMEOUT);
      sh.abort_flag = 1;
    }
    // Drain: every copy started here has landed before the CTA can leave.
    for (int i = xi > Cf::XS ? xi - Cf::XS : 0; i < xi; ++i)
      if (!mbar_wait(&sh.xfull[i % Cf::XS], (i / Cf::XS) & 1)) raise_error(err, ERR_TIMEOUT);
    for (int i = wi > Cf::WS ? wi - Cf::WS : 0; i < wi; ++i)
      if (!mbar_wait(&sh.wfull[i % Cf::WS], (i / Cf::WS) & 1)) raise_error(err, ERR_TIMEOUT);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(RT_BM, EC);
    bool ok = true;
    for (int kb = 0; kb < KB && ok; ++kb) {
      const int xs = kb % Cf::XS;
      if (!mbar_wait(&sh.xfull[xs], (kb / Cf::XS) & 1)) { ok = false; break; }
      for (int s = 0; s < 3; ++s) {
        const int j = kb * 3 + s, ws = j % Cf::WS;
        if (!mbar_wait(&sh.wfull[ws], (j / Cf::WS) & 1)) { ok = false; break; }
        if (sh.abort_flag) { ok = false; break; }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sX + xs * Cf::X_BYTES);
        const uint32_t b0 = smem_u32(sW + ws * Cf::W_BYTES);
        const uint32_t acc = s == 0 ? tmem : tmem + EC;
#pragma unroll
        for (int k = 0; k < RT_BK / 16; ++k)
          tc_mma_bf16(acc, sw128_kmajor_desc(a0 + k * 32), sw128_kmajor_desc(b0 + k * 32), idesc,
                      (kb > 0 || k > 0 || s == 2) ? 1u : 0u);
        tc_commit(&sh.wempty[ws]);
      }
      if (ok) tc_commit(&sh.xempty[xs]);
    }
    if (!ok) {
      raise_error(err, ERR_TIMEOUT);
      sh.abort_flag = 1;
    }
    tc_commit(&sh.accb);  // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // ---------------- epilogue
  if (!mbar_wait(&sh.accb, 0)) {
    raise_error(err, ERR_TIMEOUT);
    sh.abort_flag = 1;
  }
  tc_fence_after();
  __syncthreads();
  const bool run = sh.abort_flag == 0;

  const int i = warp * 32 + lane;
  const bool valid = t0 + i < T;
  const long long tok = tok0 + i;
  const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);

  // pass 1: local max / argmax (increasing e, strict >: the lowest index wins a tie), local sum
  float m = -INFINITY, ssum = 0.f;
  int a = INT_MAX;
  if (run) {
#pragma unroll 1
    for (int c0 = 0; c0 < EC; c0 += 16) {
      uint32_t h[16], r[16];
      tmem_ld16(trow + c0, h);
      tmem_ld16(trow + EC + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = e0 + c0 + j;
        if (e < E) {
          const float z = (__uint_as_float(h[j]) + __uint_as_float(r[j])) + sh.bias[c0 + j];
          if (z > m) { m = z; a = e; }
          if (logits && valid) logits[tok * E + e] = z;
        }
      }
    }
#pragma unroll 1
    for (int c0 = 0; c0 < EC; c0 += 16) {
      uint32_t h[16], r[16];
      tmem_ld16(trow + c0, h);
      tmem_ld16(trow + EC + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = e0 + c0 + j;
        if (e < E) ssum += expf((__uint_as_float(h[j]) + __uint_as_float(r[j])) + sh.bias[c0 + j] - m);
      }
    }
  }
  sh.m[i] = m;
  sh.s[i] = ssum;
  sh.a[i] = a;

  // exchange between the cluster's CTAs (expert slices in rank order)
  if (Q > 1) cluster_sync();
  float M = m, S = ssum;
  int A = a;
  if (Q > 1) {
    M = -INFINITY;
    A = INT_MAX;
    for (int rk = 0; rk < Q; ++rk) {
      const float mr = dsmem_ld_f32(dsmem_addr(&sh.m[i], rk));
      if (mr > M) {
        M = mr;
        A = dsmem_ld_s32(dsmem_addr(&sh.a[i], rk));
      }
    }
    S = 0.f;
    for (int rk = 0; rk < Q; ++rk) {
      const float mr = dsmem_ld_f32(dsmem_addr(&sh.m[i], rk));
      const float sr = dsmem_ld_f32(dsmem_addr(&sh.s[i], rk));
      if (sr > 0.f) S += sr * expf(mr - M);
    }
  }
  if (A < 0 || A >= E) {  // only non-finite logits (or an aborted tile) get here
    if (run && valid) raise_error(err, ERR_BOUNDS);
    A = 0;
  }
  sh.texp[i] = valid ? A : -1;

  // pass 2: probabilities and their column sums over the tile
#pragma unroll 1
  for (int c0 = 0; c0 < EC; c0 += 16) {
    float p[16];
    if (run) {
      uint32_t h[16], r[16];
      tmem_ld16(trow + c0, h);
      tmem_ld16(trow + EC + c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int e = e0 + c0 + j;
        const float z = (__uint_as_float(h[j]) + __uint_as_float(r[j])) + sh.bias[c0 + j];
        p[j] = (valid && e < E) ? expf(z - M) / S : 0.f;
        if (probs && valid && e < E) probs[tok * E + e] = p[j];
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) p[j] = 0.f;
    }
    const float cs = warp_colsum16(p, lane);
    if ((lane & 1) == 0) sh.colsum[warp][c0 + (lane >> 1)] = cs;
  }
  if (valid && A >= e0 && A < e0 + EC) atomicAdd(&sh.hist[A - e0], 1);
  __syncthreads();

  const size_t tbase = ((size_t)g * nT + tile) * E;
  for (int c = threadIdx.x; c < EC; c += blockDim.x) {
    const int e = e0 + c;
    if (e < E) {
      tile_P[tbase + e] = ((sh.colsum[0][c] + sh.colsum[1][c]) + sh.colsum[2][c]) + sh.colsum[3][c];
      tile_hist[tbase + e] = sh.hist[c];
    }
  }
  if (q == 0) {
    // rank among the tile's earlier tokens with the same expert
    const int key = valid ? A : -1 - lane;
    const unsigned same = __match_any_sync(0xffffffffu, key);
    int rk = __popc(same & ((1u << lane) - 1u));
    for (int j = 0; j < warp * 32; ++j) rk += sh.texp[j] == A;
    if (valid) {
      expert[tok] = A;
      gate[tok] = 1.0f / S;  // exp(z_A - M) / S with z_A = M; never renormalised
      rank[tok] = rk;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, Cf::TMEM_COLS);
  if (Q > 1) cluster_sync();  // peers are done reading this CTA's m / s / a
}

// ---------------------------------------------------------------- host side
template <int EC>
static int launch_rt(const CUtensorMap& tmX, const CUtensorMap& tmW, const RouteArgs& a, int nT, int Q,
                     int32_t* rank, cudaStream_t s) {
  auto kern = router_tc_kernel<EC>;
  constexpr int smem = rt_smem_bytes<EC>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(Q * nT), (unsigned)a.G, 1);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)Q;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = Q > 1 ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmX, tmW, a.br, a.T, a.E, a.d, nT, Q, a.expert, a.gate,
                                           rank, a.tile_hist, a.tile_P, a.logits_out, a.probs, a.err);
  return e == cudaSuccess ? 1 : -1;
}

// Experts per CTA: the smallest power of two >= 16 that keeps the cluster at <= 8
// CTAs, raised to 64 when E allows (more parallel CTAs for few-token batches).
int router_tc_experts_per_cta(int E) {
  int ec = 16;
  while ((E + ec - 1) / ec > 8) ec *= 2;
  int want = 16;
  while (want < E && want < 64) want *= 2;
  return ec > want ? ec : want;
}

int launch_router_tc(const RouteArgs& a, int32_t* rank, cudaStream_t s) {
  const long long N = (long long)a.G * a.T;
  if (N == 0) return 0;
  const int nT = (a.T + RT_BM - 1) / RT_BM;
  const int EC = router_tc_experts_per_cta(a.E);
  const int Q = (a.E + EC - 1) / EC;
  if (EC > 256 || Q > 8) return -1;
  const long long n = (long long)a.E * a.d;
  const unsigned sb = (unsigned)((n + 255) / 256 < 148 * 16 ? (n + 255) / 256 : 148 * 16);
  router_split_kernel<<<sb, 256, 0, s>>>(a.Wr, (__nv_bfloat16*)a.wsplit, n);
  if (cudaGetLastError() != cudaSuccess) return -1;
  CUtensorMap tmX, tmW;
  if (!encode_bf16_2d(&tmX, a.x, (uint64_t)N, (uint64_t)a.d, RT_BM)) return -1;
  if (!encode_bf16_2d(&tmW, a.wsplit, (uint64_t)3 * a.E, (uint64_t)a.d, (uint32_t)EC)) return -1;
  int n2;
  switch (EC) {
    case 16: n2 = launch_rt<16>(tmX, tmW, a, nT, Q, rank, s); break;
    case 32: n2 = launch_rt<32>(tmX, tmW, a, nT, Q, rank, s); break;
    case 64: n2 = launch_rt<64>(tmX, tmW, a, nT, Q, rank, s); break;
    case 128: n2 = launch_rt<128>(tmX, tmW, a, nT, Q, rank, s); break;
    default: n2 = launch_rt<256>(tmX, tmW, a, nT, Q, rank, s); break;
  }
  return n2 < 0 ? -1 : 2;
}

}  // namespace smoe
