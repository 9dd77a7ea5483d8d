// Router of the top-1 Switch layer on 5th-generation tensor cores (tcgen05, sm_103a).
//
// The router runs in float32 (selective precision: Switch Transformers card on
// ai-papers.xuzou.cn, 方法适配; "042 · Switch Transformer：每个词只选一个专家",
// section 一, p(x) = softmax(W_r x)).  The activations are bfloat16, so every x_k
// is exact in bfloat16; W_r is float32 and is split into three bfloat16 pieces
// hi + mid + lo whose sum equals w to within 2^-24 |w| (each piece holds the
// next 8 bits of the significand).  Then
//     z = x . hi + (x . mid + x . lo)
// with every bf16 x bf16 product exact and accumulated in float32 by the tensor
// cores, each piece in its own TMEM accumulator so the small terms never share an
// accumulator with the large ones; the pieces are added in the epilogue.
//
// One CTA (or a cluster of Q CTAs, each with EC experts) takes a tile of 128
// tokens of one routing group:
//   warp 0, one lane : TMA producer; one stage = the x tile and the slice's three
//                      W pieces for 64 or 128 columns of K, behind one barrier
//   warp 1, one lane : MMA issuer (M = 128 tokens, N = 3 EC rows of pieces, K = 16)
//   16 warps         : epilogue; warp w reads TMEM lane quadrant w % 4 (32 tokens)
//                      and column group w / 4 (a quarter of the CTA's experts):
//     pass 1  logits z (+ bias) into registers, max / argmax (ties -> lowest index),
//             combined over the column groups through shared memory
//     pass 1b exp(z - max) in registers (ex2 of the log2e-scaled difference), sums
//     exchange of (max, sum, argmax) between the Q CTAs through distributed shared memory
//     pass 2  p = exp(z - max) * exp(max - Max) / Sum; column sums over the tile's
//             tokens (warp reduce-scatter), expert histogram of the tile, rank of
//             each token among the tile's earlier tokens with the same expert.
// Outputs per token: expert (raw choice), gate = p_{expert}, rank in tile; per
// (group, tile, expert): token count and probability sum.  The cross-tile scan
// that turns ranks into slots runs in route.cu.
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int RT_BM = ROUTE_TILE;  // 128 tokens per tile
constexpr int RT_BK = 64;          // 64 bf16 = one 128-byte swizzle row
constexpr int RT_THREADS = 512;    // 16 warps: 4 TMEM lane quadrants x 4 column groups
constexpr float LOG2E = 1.4426950408889634f;

// ---------------------------------------------------------------- W_r -> hi, mid, lo
// Layout of the pieces: [Q slices][hi, mid, lo][EC experts][d], experts past E zero, so
// one TMA box (and one MMA) covers all three pieces of a slice's experts.
__global__ void router_split_kernel(const float* __restrict__ Wr, __nv_bfloat16* __restrict__ ws, int E, int d,
                                    int EC, long long n /* Q * EC * d */) {
  griddep_wait();
  griddep_launch_dependents();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / d;  // q * EC + el = expert index
    const int k = (int)(i - row * d);
    const int q = (int)(row / EC), el = (int)(row - (long long)q * EC);
    const float w = row < E ? Wr[row * d + k] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);  // exact: fits in the 24-bit significand
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);  // exact
    const size_t base = ((size_t)q * 3 * EC + el) * d + k;
    ws[base] = hi;
    ws[base + (size_t)EC * d] = mid;
    ws[base + (size_t)2 * EC * d] = __float2bfloat16_rn(r2);
  }
}

// ---------------------------------------------------------------- tiling
// Per 64-column atom of K, a stage holds the x tile (128 tokens) and the 3 * EC rows of
// W pieces of the CTA's slice, in WBOXES boxes of MMA_N rows; MMA m takes box m.
// Accumulators in TMEM: one block of EC columns per piece (hi, mid, lo); with EC = 256
// the 512 columns hold hi and (mid + lo).
template <int EC>
struct RtGeom {
  static constexpr int WROWS = 3 * EC;
  static constexpr int MMA_N = EC == 256 ? 256 : (WROWS <= 256 ? WROWS : 192);
  static constexpr int WBOXES = WROWS / MMA_N;
  static constexpr int ACC_BLOCKS = EC == 256 ? 2 : 3;
  static constexpr uint32_t TMEM_COLS = ACC_BLOCKS * EC <= 32 ? 32 : ACC_BLOCKS * EC <= 64 ? 64
                                       : ACC_BLOCKS * EC <= 128 ? 128 : ACC_BLOCKS * EC <= 256 ? 256 : 512;
  // first TMEM column written by MMA m
  static __device__ __forceinline__ uint32_t dcol(int m) { return EC == 256 ? (m == 0 ? 0u : 256u) : (uint32_t)(m * MMA_N); }
  static_assert(WROWS % MMA_N == 0 && MMA_N % 16 == 0 && MMA_N <= 256, "tcgen05 M=128 takes N = 16..256, step 16");
  static_assert((MMA_N * 128) % 1024 == 0, "every W box starts on a swizzle atom");
};

// DEEP: one CTA per SM with ~170-220 KB of loads in flight (a grid that fits in one
// wave); !DEEP: two CTAs per SM (each <= 113 KB, <= 256 TMEM columns), so one CTA's
// epilogue overlaps the other's main loop on larger grids.  Each stage is one barrier
// phase: per-phase cost, not bytes, limits a CTA's TMA stream, so stages are large.
template <int EC, bool DEEP>
struct RtCfg {
  using G = RtGeom<EC>;
  static constexpr int NA = (EC <= 16 || (EC <= 64 && DEEP)) ? 2 : 1;  // 64-column atoms per stage
  static constexpr int X_ATOM = RT_BM * RT_BK * 2;                    // 16 KB
  static constexpr int W_ATOM = G::WROWS * RT_BK * 2;
  static constexpr int STAGE_BYTES = NA * (X_ATOM + W_ATOM);
  static constexpr int RING_BUDGET = DEEP ? 224 * 1024 : 110 * 1024;
  static constexpr int STAGES = RING_BUDGET / STAGE_BYTES < 4 ? RING_BUDGET / STAGE_BYTES : 4;
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static_assert(STAGES >= 2, "double buffering at least");
  static_assert(DEEP || G::TMEM_COLS <= 256, "two CTAs per SM share the 512 TMEM columns");
  static_assert(NA == 1 || G::WBOXES == 1, "a 3-D W box spans atoms only when one box covers the pieces");
};

template <int EC, bool DEEP>
struct RtBars {
  uint64_t full[RtCfg<EC, DEEP>::STAGES], empty[RtCfg<EC, DEEP>::STAGES];
  uint64_t accb;
  uint32_t tmem_slot;
  volatile int abort_flag;
};

// Epilogue scratch; it reuses the ring's shared memory once every MMA has completed.
template <int EC>
struct RtScratch {
  float red_m[4][RT_BM];  // per column group: max logit of each token
  int red_a[4][RT_BM];    // per column group: argmax
  float red_s[4][RT_BM];  // per column group: sum of exp(z - m)
  float m[RT_BM];         // this CTA's experts: max logit per token (read by cluster peers)
  float s[RT_BM];         // this CTA's experts: sum of exp(z - m)
  int a[RT_BM];           // this CTA's experts: argmax
  float Mall[RT_BM];      // all experts: max logit per token
  float Sall[RT_BM];      // all experts: sum of exp(z - Mall)
  int texp[RT_BM];        // final expert per token (-1 past the group's end)
  float zz[RT_BM];        // (log sum_e exp z)^2 per token (0 past the group's end)
  float colsum[4][EC];    // per lane quadrant: probability sums of the columns
  int hist[EC];
  float bias[EC];
};

template <int EC, bool DEEP>
constexpr int rt_smem_bytes() {
  return RtCfg<EC, DEEP>::RING_BYTES + (int)sizeof(RtBars<EC, DEEP>) + 1024;
}
static_assert(sizeof(RtScratch<256>) <= RtCfg<256, true>::RING_BYTES, "scratch fits in the ring");
static_assert(sizeof(RtScratch<16>) <= RtCfg<16, false>::RING_BYTES, "scratch fits in the ring");
static_assert(rt_smem_bytes<256, true>() <= 227 * 1024 && rt_smem_bytes<128, true>() <= 227 * 1024 &&
                  rt_smem_bytes<64, true>() <= 227 * 1024 && rt_smem_bytes<32, true>() <= 227 * 1024 &&
                  rt_smem_bytes<16, true>() <= 227 * 1024,
              "deep ring fits in one SM's shared memory");
static_assert(rt_smem_bytes<64, false>() <= 113 * 1024 && rt_smem_bytes<32, false>() <= 113 * 1024 &&
                  rt_smem_bytes<16, false>() <= 113 * 1024,
              "shallow ring lets two CTAs share an SM");

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
template <int EC, bool DEEP>
__global__ void __launch_bounds__(RT_THREADS, DEEP ? 1 : 2)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const float* __restrict__ br, int T, int E, int d, int nT, int Q, int use3d,
                     int32_t* __restrict__ expert, float* __restrict__ gate, int32_t* __restrict__ rank,
                     int32_t* __restrict__ tile_hist, float* __restrict__ tile_P, float* __restrict__ tile_Z,
                     float* __restrict__ logits, float* __restrict__ probs, uint32_t* err) {
  using Cf = RtCfg<EC, DEEP>;
  using Gm = RtGeom<EC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RtBars<EC, DEEP>& bar = *reinterpret_cast<RtBars<EC, DEEP>*>(smem + Cf::RING_BYTES);
  RtScratch<EC>& sh = *reinterpret_cast<RtScratch<EC>*>(smem);  // valid after the main loop

  const int q = Q > 1 ? (int)cluster_ctarank() : 0;
  const int tile = blockIdx.x / Q;
  const int g = blockIdx.y;
  const int e0 = q * EC;
  const int t0 = tile * RT_BM;
  const long long tok0 = (long long)g * T + t0;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NST = (d + Cf::NA * RT_BK - 1) / (Cf::NA * RT_BK);  // stages along K

  if (threadIdx.x == 0) {
    for (int i = 0; i < Cf::STAGES; ++i) {
      mbar_init(&bar.full[i], 1);
      mbar_init(&bar.empty[i], 1);
    }
    mbar_init(&bar.accb, 1);
    bar.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(&bar.tmem_slot, Gm::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_slot;
  griddep_launch_dependents();  // after the TMEM allocation: a dependent grid cannot starve it

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    int issued = 0;
    bool ok = true;
    griddep_wait();  // the W_r pieces come from the previous kernel
    for (int st = 0; st < NST; ++st) {
      const int slot = st % Cf::STAGES;
      if (st >= Cf::STAGES && !mbar_wait(&bar.empty[slot], ((st / Cf::STAGES) - 1) & 1)) { ok = false; break; }
      if (bar.abort_flag) { ok = false; break; }
      uint8_t* stage = smem + slot * Cf::STAGE_BYTES;
      if (use3d) {
        // one 3-D box per operand covers the stage's NA atoms (past d: zeros, not used)
        mbar_arrive_expect_tx(&bar.full[slot], (uint32_t)Cf::STAGE_BYTES);
        tma_load_3d(stage, &tmX, &bar.full[slot], 0, (int)tok0, st * Cf::NA);
        for (int b = 0; b < Gm::WBOXES; ++b)  // WBOXES > 1 only with NA = 1
          tma_load_3d(stage + Cf::NA * Cf::X_ATOM + b * Gm::MMA_N * 128, &tmW, &bar.full[slot], 0,
                      q * Gm::WROWS + b * Gm::MMA_N, st * Cf::NA);
      } else {
        const int na = min(Cf::NA, (d - st * Cf::NA * RT_BK + RT_BK - 1) / RT_BK);  // atoms inside d
        mbar_arrive_expect_tx(&bar.full[slot], (uint32_t)(na * (Cf::X_ATOM + Cf::W_ATOM)));
        for (int at = 0; at < na; ++at) {
          const int kx = (st * Cf::NA + at) * RT_BK;
          tma_load_2d(stage + at * Cf::X_ATOM, &tmX, &bar.full[slot], kx, (int)tok0);
          for (int b = 0; b < Gm::WBOXES; ++b)
            tma_load_2d(stage + Cf::NA * Cf::X_ATOM + at * Cf::W_ATOM + b * Gm::MMA_N * 128, &tmW, &bar.full[slot],
                        kx, q * Gm::WROWS + b * Gm::MMA_N);
        }
      }
      issued = st + 1;
    }
    if (!ok) {
      raise_error(err, ERR_TIMEOUT);
      bar.abort_flag = 1;
    }
    // Drain: every copy started here has landed before the CTA can leave.
    for (int i = issued > Cf::STAGES ? issued - Cf::STAGES : 0; i < issued; ++i)
      if (!mbar_wait(&bar.full[i % Cf::STAGES], (i / Cf::STAGES) & 1)) raise_error(err, ERR_TIMEOUT);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(RT_BM, Gm::MMA_N);
    bool ok = true;
    for (int st = 0; st < NST && ok; ++st) {
      const int slot = st % Cf::STAGES;
      if (!mbar_wait(&bar.full[slot], (st / Cf::STAGES) & 1)) { ok = false; break; }
      if (bar.abort_flag) { ok = false; break; }
      tc_fence_after();
      const int na = min(Cf::NA, (d - st * Cf::NA * RT_BK + RT_BK - 1) / RT_BK);
      const uint32_t stage = smem_u32(smem + slot * Cf::STAGE_BYTES);
      for (int at = 0; at < na; ++at) {
        const uint32_t xa = stage + at * Cf::X_ATOM;
        const uint32_t wa = stage + Cf::NA * Cf::X_ATOM + at * Cf::W_ATOM;
#pragma unroll
        for (int kk = 0; kk < RT_BK / 16; ++kk)
#pragma unroll
          for (int mm = 0; mm < Gm::WBOXES; ++mm) {
            const bool first = st == 0 && at == 0 && kk == 0 && !(EC == 256 && mm == 2);
            tc_mma_bf16(tmem + Gm::dcol(mm), sw128_kmajor_desc(xa + kk * 32),
                        sw128_kmajor_desc(wa + mm * Gm::MMA_N * 128 + kk * 32), idesc, first ? 0u : 1u);
          }
      }
      tc_commit(&bar.empty[slot]);
    }
    if (!ok) {
      raise_error(err, ERR_TIMEOUT);
      bar.abort_flag = 1;
    }
    tc_commit(&bar.accb);  // arrives once every MMA issued above has completed
  }
  __syncwarp();

  // ---------------- epilogue
  if (!mbar_wait(&bar.accb, 0)) {
    raise_error(err, ERR_TIMEOUT);
    bar.abort_flag = 1;
  }
  tc_fence_after();
  __syncthreads();  // every MMA has read its operands: the ring is scratch from here on
  const bool run = bar.abort_flag == 0;
  for (int c = threadIdx.x; c < EC; c += blockDim.x) {
    const int e = e0 + c;
    sh.bias[c] = (br && e < E) ? br[e] : 0.f;
    sh.hist[c] = 0;
  }
  __syncthreads();

  // Warp w reads TMEM lane quadrant lq = w % 4 (tokens 32 lq .. 32 lq + 31) and column
  // group cg = w / 4 (CPW consecutive experts); NCG groups cover the CTA's EC experts.
  constexpr int NCG = EC >= 64 ? 4 : EC / 16;
  constexpr int CPW = EC / NCG;
  const int lq = warp & 3, cg = warp >> 2;
  const bool has_cols = cg < NCG;
  const int cbeg = cg * CPW;
  const int i = lq * 32 + lane;
  const bool valid = t0 + i < T;
  const long long tok = tok0 + i;
  const uint32_t trow = tmem + ((uint32_t)(lq * 32) << 16);

  // pass 1: logits z (+ bias) into registers; max / argmax over this warp's columns
  // (increasing e with strict >, so the lowest index wins a tie)
  float v[CPW];
  float m = -INFINITY;
  int a = INT_MAX;
  if (run && has_cols) {
#pragma unroll
    for (int ch = 0; ch < CPW / 16; ++ch) {
      const uint32_t col = (uint32_t)(cbeg + ch * 16);
      uint32_t h[16], r1[16], r2[16];
      tmem_ld16(trow + col, h);
      tmem_ld16(trow + EC + col, r1);
      if (Gm::ACC_BLOCKS == 3) tmem_ld16(trow + 2 * EC + col, r2);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = cbeg + ch * 16 + j;
        const float corr = Gm::ACC_BLOCKS == 3 ? __uint_as_float(r1[j]) + __uint_as_float(r2[j])
                                                : __uint_as_float(r1[j]);
        const float z = (__uint_as_float(h[j]) + corr) + sh.bias[c];
        v[ch * 16 + j] = z;
        if (e0 + c < E) {
          if (z > m) { m = z; a = e0 + c; }
        }
      }
      if (logits && valid) {  // the chunk's 16 logits of this token: 16-byte stores when aligned
        const int c0 = e0 + cbeg + ch * 16;
        float* dst = logits + tok * E + c0;
        if ((E & 3) == 0 && c0 + 16 <= E) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            *reinterpret_cast<float4*>(dst + 4 * q4) =
                make_float4(v[ch * 16 + 4 * q4], v[ch * 16 + 4 * q4 + 1], v[ch * 16 + 4 * q4 + 2],
                            v[ch * 16 + 4 * q4 + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < E) dst[j] = v[ch * 16 + j];
        }
      }
    }
  }
  if (has_cols) {
    sh.red_m[cg][i] = m;
    sh.red_a[cg][i] = a;
  }
  __syncthreads();
  float mc = -INFINITY;  // max over this CTA's experts
  int ac = INT_MAX;
#pragma unroll
  for (int k = 0; k < NCG; ++k)
    if (sh.red_m[k][i] > mc) { mc = sh.red_m[k][i]; ac = sh.red_a[k][i]; }

  // pass 1b: exp(z - mc) in registers, partial sums
  float ps = 0.f;
  if (run && has_cols) {
    const float mcs = mc * LOG2E;
#pragma unroll
    for (int k = 0; k < CPW; ++k) {
      const float ex = (e0 + cbeg + k < E) ? ex2_approx(fmaf(v[k], LOG2E, -mcs)) : 0.f;
      v[k] = ex;
      ps += ex;
    }
  }
  if (has_cols) sh.red_s[cg][i] = ps;
  __syncthreads();
  if (cg == 0) {
    float sc = 0.f;
#pragma unroll
    for (int k = 0; k < NCG; ++k) sc += sh.red_s[k][i];
    sh.m[i] = mc;
    sh.s[i] = sc;
    sh.a[i] = ac;
  }

  // exchange between the cluster's CTAs (expert slices in rank order)
  if (Q > 1) cluster_sync();
  else __syncthreads();
  if (cg == 0) {
    float M = sh.m[i], S = sh.s[i];
    int A = sh.a[i];
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
    sh.Mall[i] = M;
    sh.Sall[i] = S;
    sh.texp[i] = valid ? A : -1;
    const float lse = M + logf(S);  // log sum_e exp z_e over all E experts (router z-loss)
    sh.zz[i] = (run && valid) ? lse * lse : 0.f;
  }
  __syncthreads();

  // pass 2: p = exp(z - mc) * exp(mc - M) / S; column sums over the tile's tokens
  const float scale = (run && valid) ? expf(mc - sh.Mall[i]) / sh.Sall[i] : 0.f;
  if (has_cols) {
#pragma unroll
    for (int ch = 0; ch < CPW / 16; ++ch) {
      float p[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = cbeg + ch * 16 + j;
        p[j] = v[ch * 16 + j] * scale;  // 0 past E (v = 0) and for invalid tokens (scale = 0)
        if (probs && valid && run && e0 + c < E) probs[tok * E + e0 + c] = p[j];
      }
      const float cs = warp_colsum16(p, lane);
      if ((lane & 1) == 0) sh.colsum[lq][cbeg + ch * 16 + (lane >> 1)] = cs;
    }
  }
  const int A = sh.texp[i];
  if (cg == 0 && A >= e0 && A < e0 + EC) atomicAdd(&sh.hist[A - e0], 1);
  __syncthreads();

  const size_t tbase = ((size_t)g * nT + tile) * E;
  if (q == 0 && warp == 0) {  // the tile's sum of (log sum exp z)^2, fixed order
    float zs = (sh.zz[lane] + sh.zz[lane + 32]) + (sh.zz[lane + 64] + sh.zz[lane + 96]);
    zs = warp_sum(zs);
    if (lane == 0) tile_Z[(size_t)g * nT + tile] = zs;
  }
  for (int c = threadIdx.x; c < EC; c += blockDim.x) {
    const int e = e0 + c;
    if (e < E) {
      tile_P[tbase + e] = ((sh.colsum[0][c] + sh.colsum[1][c]) + sh.colsum[2][c]) + sh.colsum[3][c];
      tile_hist[tbase + e] = sh.hist[c];
    }
  }
  if (q == 0 && cg == 0) {
    // rank among the tile's earlier tokens with the same expert
    const int key = valid ? A : -1 - lane;
    const unsigned same = __match_any_sync(0xffffffffu, key);
    int rk = __popc(same & ((1u << lane) - 1u));
    for (int j = 0; j < lq * 32; ++j) rk += sh.texp[j] == A;
    if (valid) {
      expert[tok] = A;
      gate[tok] = 1.0f / sh.Sall[i];  // exp(z_A - M) / S with z_A = M; never renormalised
      rank[tok] = rk;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, Gm::TMEM_COLS);
  if (Q > 1) cluster_sync();  // peers are done reading this CTA's m / s / a
}

// ---------------------------------------------------------------- host side
template <int EC, bool DEEP>
static int launch_rt(const CUtensorMap& tmX, const CUtensorMap& tmW, const RouteArgs& a, int nT, int Q, int use3d,
                     int32_t* rank, cudaStream_t s) {
  auto kern = router_tc_kernel<EC, DEEP>;
  constexpr int smem = rt_smem_bytes<EC, DEEP>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1;
  const cudaError_t e = launch_k(kern, dim3((unsigned)(Q * nT), (unsigned)a.G, 1), dim3(RT_THREADS, 1, 1), smem, s,
                                 /*pdl=*/true, (unsigned)Q, tmX, tmW, a.br, a.T, a.E, a.d, nT, Q, use3d, a.expert,
                                 a.gate, rank, a.tile_hist, a.tile_P, a.tile_Z, a.logits_out, a.probs, a.err);
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

int router_tc_mma_n(int EC) { return EC == 256 ? 256 : (3 * EC <= 256 ? 3 * EC : 192); }

size_t router_tc_wsplit_bytes(int E, int d) {
  const int EC = router_tc_experts_per_cta(E);
  const size_t Q = (size_t)((E + EC - 1) / EC);
  return Q * EC * 3 * (size_t)d * 2;
}

int launch_router_tc(const RouteArgs& a, int32_t* rank, cudaStream_t s) {
  const long long N = (long long)a.G * a.T;
  if (N == 0) return 0;
  const int nT = (a.T + RT_BM - 1) / RT_BM;
  const int EC = router_tc_experts_per_cta(a.E);
  const int Q = (a.E + EC - 1) / EC;
  if (EC > 256 || Q > 8) return -1;
  const long long n = (long long)Q * EC * a.d;
  const unsigned sb = (unsigned)((n + 255) / 256 < 148 * 16 ? (n + 255) / 256 : 148 * 16);
  if (launch_k(router_split_kernel, dim3(sb), dim3(256), 0, s, false, 1, a.Wr, (__nv_bfloat16*)a.wsplit, a.E, a.d, EC,
               n) != cudaSuccess)
    return -1;
  // One wave on this device's SMs -> the deep ring; EC >= 128 always takes it (512 TMEM columns).
  const long long ctas = (long long)Q * nT * a.G;
  const bool deep = EC >= 128 || ctas <= (long long)device_sm_count();
  const int NA = (EC <= 16 || (EC <= 64 && deep)) ? 2 : 1;  // RtCfg<EC, deep>::NA
  const int use3d = a.d % RT_BK == 0 ? 1 : 0;
  CUtensorMap tmX, tmW;
  if (use3d) {
    if (!encode_bf16_3d(&tmX, a.x, (uint64_t)N, (uint64_t)a.d, RT_BM, (uint32_t)NA)) return -1;
    if (!encode_bf16_3d(&tmW, a.wsplit, (uint64_t)3 * Q * EC, (uint64_t)a.d, (uint32_t)router_tc_mma_n(EC),
                        (uint32_t)NA))
      return -1;
  } else {
    if (!encode_bf16_2d(&tmX, a.x, (uint64_t)N, (uint64_t)a.d, RT_BM)) return -1;
    if (!encode_bf16_2d(&tmW, a.wsplit, (uint64_t)3 * Q * EC, (uint64_t)a.d, (uint32_t)router_tc_mma_n(EC)))
      return -1;
  }
  int n2;
#define SMOE_RT(ECV)                                                                                        \
  n2 = deep ? launch_rt<ECV, true>(tmX, tmW, a, nT, Q, use3d, rank, s)                                      \
            : launch_rt<ECV, false>(tmX, tmW, a, nT, Q, use3d, rank, s)
  switch (EC) {
    case 16: SMOE_RT(16); break;
    case 32: SMOE_RT(32); break;
    case 64: SMOE_RT(64); break;
    case 128: n2 = launch_rt<128, true>(tmX, tmW, a, nT, Q, use3d, rank, s); break;
    default: n2 = launch_rt<256, true>(tmX, tmW, a, nT, Q, use3d, rank, s); break;
  }
#undef SMOE_RT
  return n2 < 0 ? -1 : 2;
}

}  // namespace smoe
