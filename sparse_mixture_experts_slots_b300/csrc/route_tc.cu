// Router of the Switch layer on 5th-generation tensor cores (tcgen05, sm_103a).
//
// The router runs in float32 (selective precision: Switch Transformers card on
// ai-papers.xuzou.cn, 方法适配; "042 · Switch Transformer：每个词只选一个专家",
// section 一, p(x) = softmax(W_r x)).  The activations are bfloat16, so every x_k
// is exact in bfloat16; W_r is float32 and is split into three bfloat16 pieces
// hi + mid + lo whose sum equals w to within 2^-24 |w| (each piece holds the
// next 8 bits of the significand).  Then
//     z = x . hi + (x . mid + x . lo)
// with every bf16 x bf16 product exact and accumulated in float32 by the tensor
// cores, the hi piece in its own TMEM accumulator so the small terms never share an
// accumulator with the large ones; the pieces are added in the epilogue.
//
// One persistent kernel; a work item is one token tile (128 tokens of one routing group)
// times one slice of EC experts (slice q: experts q EC .. q EC + EC - 1), Q slices per tile.
// Two ways to put the slices of a tile together:
//   clusters  a cluster of Q CTAs (CTA q holds slice q) walks the tiles; clusters take tiles
//             in turn; the per-token partials move through distributed shared memory.
//             Clusters of 4 or 8 CTAs fit on fewer SMs (8: 120 of 148), so this is used for
//             Q <= 2 (and where no exchange buffer is given);
//   global    every SM runs one CTA of a cooperative grid; CTA c takes items c, c + grid, ...
//             (item = tile Q + slice); the partials go through global memory, each slice's
//             flag set to the launch's epoch when they are written.  An item waits only on the
//             other slices of its tile, items a CTA owns come in increasing order, and the
//             slices of a tile are items within Q - 1 of each other, so every wait is on work
//             that is running or done.  The epoch lives in device memory: every CTA reads it
//             at the start, and the last CTA to finish advances it (a ticket), so a replayed
//             CUDA graph of the call still sees a fresh epoch.
// Per CTA:
//   warp 0, one lane : TMA producer.  Per 64-column atom of K the x tile (an x stage holds
//                      NAX atoms) and the slice's W box(es) (hi, mid, lo rows), each in a
//                      ring slot of its own behind one barrier.
//   warp 1, one lane : MMA issuer (M = 128 tokens, N = MMA_N rows of pieces, K = 16) into
//                      one of NBUF TMEM accumulator sets; the next tile's MMAs start as soon
//                      as the epilogue has read the previous accumulator out of TMEM.
//   warps 2 .. 17    : epilogue; warp w reads TMEM lane quadrant w % 4 (32 tokens) and
//                      column group (w - 2) / 4 (a quarter of the CTA's experts):
//     pass 1  logits z (+ bias) into registers, then the accumulator is released;
//             max / argmax (ties -> lowest index), combined over the column groups
//     pass 1b exp(z - max) in registers (ex2 of the log2e-scaled difference), sums
//     exchange of (max, sum, argmax) between the Q slices: (clusters) each CTA writes its
//             values into every peer's receive buffer with asynchronous remote stores that
//             count their bytes on the peer's barrier, everyone reads the Q slices from its
//             own memory; (global) each CTA writes them to the tile's exchange rows and
//             releases its flag, then reads all Q slices once every flag carries the epoch
//     pass 2  p = exp(z - max) * exp(max - Max) / Sum; column sums over the tile's tokens
//             (warp reduce-scatter), expert histogram of the tile, rank of each token
//             among the tile's earlier tokens with the same expert.
// Outputs per token: expert (raw choice), gate = p_{expert}, rank in tile; per
// (group, tile, expert): token count and probability sum.  The cross-tile scan
// that turns ranks into slots runs in route.cu.
// Top-2 variant (T2, clusters or the global exchange, CTA pairs for 256-expert slices): the
// second-highest logit and its expert ride along through pass 1, the column-group merge and
// the exchange ("混合专家", world.lapla.si/zh/moe, 路由器只开两条线: the two highest
// scores, weighted by the softmax over those two); the outputs add the second choice, its
// gate and in-tile rank and the per-tile counts of second choices.
#include <limits.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int RT_BM = ROUTE_TILE;  // 128 tokens per tile
constexpr int RT_BK = 64;          // 64 bf16 = one 128-byte swizzle row
constexpr int RT_EPI_WARPS = 16;   // 4 TMEM lane quadrants x 4 column groups
constexpr int RT_THREADS = 64 + 32 * RT_EPI_WARPS;
constexpr int RT_RING = 192 * 1024;
constexpr int RT_MAX_WS = 8;
constexpr float LOG2E = 1.4426950408889634f;

// ---------------------------------------------------------------- W_r -> hi, mid, lo
// Layout of the pieces: [Q slices][NK atoms][hi, mid, lo][EC experts][64 columns] (experts
// past E and columns past d zero), so the W box of one MMA (MMA_N rows of one atom) is one
// contiguous block of MMA_N * 128 bytes.
__global__ void router_split_kernel(const float* __restrict__ Wr, __nv_bfloat16* __restrict__ ws, int E, int d,
                                    int EC, int NK, long long n /* Q * EC * NK * 64 */) {
  griddep_wait();
  griddep_launch_dependents();
  const int dp = NK * 64;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / dp;  // q * EC + el = expert index
    const int kd = (int)(i - row * dp);
    const int q = (int)(row / EC), el = (int)(row - (long long)q * EC);
    const int k = kd >> 6, kc = kd & 63;
    const float w = (row < E && kd < d) ? Wr[row * d + kd] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);  // exact: fits in the 24-bit significand
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);  // exact
    const size_t base = (((size_t)q * NK + k) * 3 * EC + el) * 64 + kc;
    ws[base] = hi;
    ws[base + (size_t)EC * 64] = mid;
    ws[base + (size_t)2 * EC * 64] = __float2bfloat16_rn(r2);
  }
}

// ---------------------------------------------------------------- tiling
// A W box holds MMA_N rows of the slice's pieces for one 64-column atom; MMA b takes box b.
// Accumulators in TMEM per tile: one block of EC columns per piece (hi, mid, lo); with
// EC = 256 the 512 columns hold hi and (mid + lo), one tile at a time, or (ONE) all three
// pieces go into one block of 256 columns, so two tiles' sets fit and the MMAs of the next
// tile need not wait for the epilogue.  ONE trades precision for that: the tensor cores'
// float32 sums then take the small pieces' terms at the size of the whole logit, and the
// largest logit error grows with d about 2.5 times (measured against float64: 8.0e-6 at
// d = 1024, 6.5e-6 at d = 768, against 2.5e-6 at d = 768 with hi apart), so it is used only
// where d <= 1024.
template <int EC, bool ONE = false>
struct RtGeom {
  static_assert(!ONE || EC == 256, "one accumulator block: 256-expert slices");
  static constexpr int WROWS = 3 * EC;
  static constexpr int MMA_N = EC == 256 ? 256 : (WROWS <= 256 ? WROWS : 192);
  static constexpr int WBOXES = WROWS / MMA_N;
  static constexpr int ACC_BLOCKS = ONE ? 1 : EC == 256 ? 2 : 3;
  static constexpr int TILE_COLS = ACC_BLOCKS * EC;
  static constexpr int NBUF = 2 * TILE_COLS <= 512 ? 2 : 1;
  static constexpr int COLS = NBUF * TILE_COLS;
  static constexpr uint32_t TMEM_COLS = COLS <= 32 ? 32 : COLS <= 64 ? 64 : COLS <= 128 ? 128 : COLS <= 256 ? 256 : 512;
  static constexpr int W_BOX = MMA_N * RT_BK * 2;
  // first TMEM column (within a tile's set) written by MMA b
  static __device__ __forceinline__ uint32_t dcol(int b) {
    return ONE ? 0u : EC == 256 ? (b == 0 ? 0u : 256u) : (uint32_t)(b * MMA_N);
  }
  static_assert(WROWS % MMA_N == 0 && MMA_N % 16 == 0 && MMA_N <= 256, "tcgen05 M=128 takes N = 16..256, step 16");
  static_assert(W_BOX % 1024 == 0, "every W box starts on a swizzle atom");
  static_assert(TILE_COLS <= 512, "a tile's accumulators fit in TMEM");
};

// NAX: 64-column atoms per x stage (2 when d % 128 == 0: one 3-D box of 256 bytes per row).
// PAIR: a CTA pair shares every W box, each CTA holding half of its rows.
// T2: with 256-expert slices the top-2 scratch takes the place of one W stage.
template <int EC, int NAX, bool PAIR = false, bool T2 = false>
struct RtCfg {
  using G = RtGeom<EC>;
  static constexpr int X_ATOM = RT_BM * RT_BK * 2;  // 16 KB
  static constexpr int X_STAGE = NAX * X_ATOM;
  static constexpr int XS = NAX == 2 ? 2 : 3;        // x stages
  static constexpr int WB = PAIR ? G::W_BOX / 2 : G::W_BOX;  // bytes of one W slot
  static constexpr int WS_FIT = (RT_RING - XS * X_STAGE) / WB - (T2 && EC == 256 ? 1 : 0);
  static constexpr int WS = WS_FIT < RT_MAX_WS ? WS_FIT : RT_MAX_WS;  // W stages
  static constexpr int X_BYTES = XS * X_STAGE;
  static constexpr int RING_BYTES = X_BYTES + WS * WB;
  static_assert(WS >= 3, "at least three W boxes in flight");
  static_assert(WB % 1024 == 0, "every W slot starts on a swizzle atom");
};

template <int XS, int WS>
struct RtBars {
  uint64_t xfull[XS], xempty[XS], wfull[WS], wempty[WS];
  uint64_t afull[2], aempty[2];    // accumulator sets: MMAs done / read out of TMEM
  uint64_t rfull, rfree;           // cluster exchange: receive buffer filled by all Q / read by all Q
  uint64_t drain;
  uint32_t tmem_slot;
  volatile int abort_flag;
  int ep_ok;                       // broadcast by the epilogue leader
};

// Epilogue scratch (outside the rings: the next tile's copies land while it is in use).
// T2 (top-2 routing): the second choices' partials, receive buffers and counts as well.
template <int EC, bool T2 = false>
struct RtScratch {
  float red_m[4][RT_BM];  // per column group: max logit of each token
  int red_a[4][RT_BM];    // per column group: argmax
  float red_s[4][RT_BM];  // per column group: sum of exp(z - m)
  float2 rms[8][RT_BM];   // receive buffer, per cluster rank: that slice's (max logit, sum of exp(z - max))
  int ra[8][RT_BM];       // and its argmax, per token
  float Mall[RT_BM];      // all experts: max logit per token
  float Sall[RT_BM];      // all experts: sum of exp(z - Mall)
  int texp[RT_BM];        // final expert per token (-1 past the group's end)
  float zz[RT_BM];        // (log sum_e exp z)^2 per token (0 past the group's end)
  float colsum[4][EC];    // per lane quadrant: probability sums of the columns
  int hist[EC];
  float bias[EC];
  float red_m2[T2 ? 4 : 1][RT_BM];  // (T2) per column group: second-highest logit and its expert
  int red_a2[T2 ? 4 : 1][RT_BM];
  int rm2[T2 ? 8 : 1][RT_BM];       // (T2) receive buffer: each slice's second logit (bits) and expert
  int ra2[T2 ? 8 : 1][RT_BM];
  float M2all[T2 ? RT_BM : 1];      // (T2) second-highest logit over all experts
  int texp2[T2 ? RT_BM : 1];        // (T2) second choice per token (-1 past the group's end)
  int hist2[T2 ? EC : 1];
};

template <int EC, int NAX, bool PAIR = false, bool T2 = false>
constexpr int rt_smem_bytes() {
  using Cf = RtCfg<EC, NAX, PAIR, T2>;
  return Cf::RING_BYTES + (int)sizeof(RtScratch<EC, T2>) + (int)sizeof(RtBars<Cf::XS, Cf::WS>) + 1024;
}
static_assert(rt_smem_bytes<256, 1>() <= 227 * 1024 && rt_smem_bytes<256, 2>() <= 227 * 1024 &&
                  rt_smem_bytes<128, 1>() <= 227 * 1024 && rt_smem_bytes<128, 2>() <= 227 * 1024 &&
                  rt_smem_bytes<64, 2>() <= 227 * 1024 && rt_smem_bytes<16, 1>() <= 227 * 1024 &&
                  rt_smem_bytes<256, 1, true>() <= 227 * 1024 && rt_smem_bytes<256, 2, true>() <= 227 * 1024,
              "rings and scratch fit in one SM's shared memory");
static_assert(rt_smem_bytes<64, 2, false, true>() <= 227 * 1024 && rt_smem_bytes<128, 2, false, true>() <= 227 * 1024 &&
                  rt_smem_bytes<256, 2, false, true>() <= 227 * 1024 && rt_smem_bytes<256, 2, true, true>() <= 227 * 1024,
              "the top-2 scratch fits too (with two-atom x stages; d % 128 != 0 keeps the separate top-2 pass)");

// Sum of p over the 32 lanes for 8 columns at once (reduce-scatter).  On return, lane L
// holds the warp's total of column (L >> 2) & 7 (lanes 4c .. 4c + 3 agree).
__device__ __forceinline__ float warp_colsum8(const float* p, int lane) {
  float v4[4], v2[2];
  const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = b4 ? p[j] : p[j + 4];
    const float keep = b4 ? p[j + 4] : p[j];
    v4[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = b3 ? v4[j] : v4[j + 2];
    const float keep = b3 ? v4[j + 2] : v4[j];
    v2[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float send = b2 ? v2[0] : v2[1];
  const float keep = b2 ? v2[1] : v2[0];
  float v1 = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
  return v1 + __shfl_xor_sync(0xffffffffu, v1, 1);
}

// (m1, a1, m2, a2) <- the two highest of (m1, a1, m2, a2) and (n1, b1, n2, b2), where every
// expert of the second pair ranks after every expert of the first (a later column group or
// slice): ties go to the first pair, i.e. to the lower expert index.
__device__ __forceinline__ void top2_merge(float& m1, int& a1, float& m2, int& a2, float n1, int b1, float n2,
                                           int b2) {
  if (n1 > m1) {
    if (m1 >= n2) {
      m2 = m1;
      a2 = a1;
    } else {
      m2 = n2;
      a2 = b2;
    }
    m1 = n1;
    a1 = b1;
  } else if (n1 > m2) {
    m2 = n1;
    a2 = b1;
  }
}

// Named barrier over the 16 epilogue warps (the producer and MMA warps do not take part).
__device__ __forceinline__ void rt_epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * RT_EPI_WARPS) : "memory"); }

// ---------------------------------------------------------------- the router kernel
// GX false: grid Q * (clusters); clusters of Q CTAs along x when Q > 1.  Cluster c takes the
// tiles c, c + clusters, ... of the G * nT tiles (tile id = group * nT + tile in group).
// XM 1 (global): a cooperative grid of one CTA per SM; CTA c takes the items c, c + grid,
// ... of the G * nT * Q items (item = tile id * Q + slice).
// XM 2 (global, CTA pairs; EC = 256): clusters of 2 on a cooperative grid; pair p takes the
// pair items p, p + pairs, ... of the ceil(G nT / 2) * Q pair items (pair item = tile pair *
// Q + slice), cluster rank r the tile 2 (tile pair) + r (a tile id past the last one reads
// zeros and writes nothing).  The even CTA issues the MMAs of both (tcgen05 cta_group::2,
// M = 256: each CTA's 128 token rows against the slice's 256 W rows, 128 of them in each
// CTA's shared memory, tmWh's boxes), so every CTA streams half of the W bytes; both CTAs'
// copies count on the even CTA's barriers, the MMAs' completions arrive on both CTAs'.
// Exchange rows (XM >= 1): xms / xam [tile id][Q][128], xflag [tile id][Q]; xctl[0] the
// epoch of the last launch, xctl[1] the finish ticket (zero between launches).
// T2 (not with CTA pairs): top-2 routing in the same pass; expert2 / gate2 / rank2 / tile_hist2
// take the second choices, gate / gate2 the softmax over the two chosen logits; with the
// slices meeting in global memory each slice's second logit and expert go through xm2 / xa2.
// ONE (256-expert slices): the three pieces in one accumulator block (see RtGeom).
template <int EC, int NAX, int XM, bool T2 = false, bool ONE = false>
__global__ void __launch_bounds__(RT_THREADS, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmWh, const float* __restrict__ br, int T, int E, int d, int nT, int Q, int total_tiles,
                     int32_t* __restrict__ expert, float* __restrict__ gate, int32_t* __restrict__ rank,
                     int32_t* __restrict__ tile_hist, float* __restrict__ tile_P, float* __restrict__ tile_Z,
                     float* __restrict__ logits, float* __restrict__ probs, uint32_t* err, float2* __restrict__ xms,
                     int* __restrict__ xam, uint32_t* __restrict__ xflag, uint32_t* __restrict__ xctl,
                     int32_t* __restrict__ expert2, float* __restrict__ gate2, int32_t* __restrict__ rank2,
                     int32_t* __restrict__ tile_hist2, float* __restrict__ xm2, int* __restrict__ xa2) {
  constexpr bool GX = XM >= 1, P2 = XM == 2;
  static_assert(!P2 || EC == 256, "CTA pairs split 256-row W boxes");
  static_assert(!T2 || XM <= 1 || EC == 256, "top-2 routing on CTA pairs: 256-expert slices");
  using Cf = RtCfg<EC, NAX, P2, T2>;
  using Gm = RtGeom<EC, ONE>;
  constexpr int XS = Cf::XS, WS = Cf::WS, NBUF = Gm::NBUF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xring = smem;
  uint8_t* wring = smem + Cf::X_BYTES;
  using Scr = RtScratch<EC, T2>;
  Scr& sh = *reinterpret_cast<Scr*>(smem + Cf::RING_BYTES);
  RtBars<XS, WS>& bar = *reinterpret_cast<RtBars<XS, WS>*>(smem + Cf::RING_BYTES + sizeof(Scr));

  // work items: (clusters) the tiles of this cluster, slice fixed by the cluster rank;
  // (global) tile it / Q, slice it % Q
  // (pairs) tile 2 (it / Q) + rank, slice it % Q
  const int qc = (!GX && Q > 1) ? (int)cluster_ctarank() : 0;
  const int prk = P2 ? (int)cluster_ctarank() : 0;
  const bool issuer = prk == 0;  // (pairs) the even CTA issues the MMAs and arms the full barriers
  const int it0 = P2 ? (int)blockIdx.x / 2 : GX ? (int)blockIdx.x : (int)blockIdx.x / Q;
  const int istep = P2 ? (int)gridDim.x / 2 : GX ? (int)gridDim.x : (int)gridDim.x / Q;
  const int n_items = P2 ? (total_tiles + 1) / 2 * Q : GX ? total_tiles * Q : total_tiles;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NK = (d + RT_BK - 1) / RT_BK;  // atoms along K
  const int NXS = (NK + NAX - 1) / NAX;    // x stages per tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < XS; ++i) {
      mbar_init(&bar.xfull[i], 1);
      mbar_init(&bar.xempty[i], 1);
    }
    for (int i = 0; i < WS; ++i) {
      mbar_init(&bar.wfull[i], 1);
      mbar_init(&bar.wempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.afull[i], 1);
      mbar_init(&bar.aempty[i], P2 ? 2 * RT_EPI_WARPS : RT_EPI_WARPS);  // (pairs) both CTAs' epilogues
    }
    mbar_init(&bar.rfull, 1);  // the leader's expect_tx; the peers' stores complete its bytes
    mbar_init(&bar.rfree, (uint32_t)Q);
    mbar_init(&bar.drain, 1);
    bar.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(P2 ? &tmWh : &tmW);
  }
  if (warp == 1) {
    if (P2) {
      tmem_alloc_pair(&bar.tmem_slot, Gm::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bar.tmem_slot, Gm::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if ((!GX && Q > 1) || P2) cluster_sync();  // every peer's barriers are initialised before any remote arrival
  const uint32_t tmem = bar.tmem_slot;
  // (global) this launch's flag value; no CTA advances xctl[0] before every CTA has read it
  const uint32_t epoch = GX ? __ldcg(xctl) + 1u : 0u;
  griddep_launch_dependents();  // after the TMEM allocation: a dependent grid cannot starve it
  // This grid may start while the previous kernel of the stream still runs: everything it
  // reads from memory (x, the W_r pieces, br) is read after this wait.
  griddep_wait();
  for (int c = threadIdx.x; c < EC; c += blockDim.x) {
    const int e = qc * EC + c;  // (global: reloaded per item)
    sh.bias[c] = e < E ? (br ? br[e] : 0.f) : -INFINITY;  // padding experts never win and weigh 0
    sh.hist[c] = 0;
    if (T2) sh.hist2[c] = 0;
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t xi = 0, wi = 0;
      bool ok = true;
      for (int it = it0; it < n_items && ok; it += istep) {
        const int q = GX ? it % Q : qc;
        const int tid = P2 ? 2 * (it / Q) + prk : GX ? it / Q : it;
        const int g = tid / nT, tile = tid - g * nT;
        const int row0 = g * T + tile * RT_BM;  // past the last tile: rows past N, read as zeros
        for (int xs = 0; xs < NXS && ok; ++xs) {
          if (bar.abort_flag) { ok = false; break; }
          const int slot = (int)(xi % XS);
          if (xi >= (uint32_t)XS && !mbar_wait(&bar.xempty[slot], ((xi / XS) - 1) & 1)) { ok = false; break; }
          if (issuer) mbar_arrive_expect_tx(&bar.xfull[slot], (uint32_t)(P2 ? 2 * Cf::X_STAGE : Cf::X_STAGE));
          if (P2) {  // counted on the even CTA's barrier
            const uint32_t xb = dsmem_addr(&bar.xfull[slot], 0);
            if (NAX == 2)
              tma_load_3d_pair(xring + slot * Cf::X_STAGE, &tmX, xb, 0, row0, xs * 2);
            else
              tma_load_2d_pair(xring + slot * Cf::X_STAGE, &tmX, xb, xs * RT_BK, row0);
          } else if (NAX == 2) {  // one 3-D box: two atoms of 128 rows (past d: zeros, never used)
            tma_load_3d(xring + slot * Cf::X_STAGE, &tmX, &bar.xfull[slot], 0, row0, xs * 2);
          } else {
            tma_load_2d(xring + slot * Cf::X_STAGE, &tmX, &bar.xfull[slot], xs * RT_BK, row0);
          }
          ++xi;
          for (int at = 0; at < NAX && ok; ++at) {
            const int k = xs * NAX + at;
            if (k >= NK) break;
            for (int b = 0; b < Gm::WBOXES; ++b) {
              const int ws = (int)(wi % WS);
              if (wi >= (uint32_t)WS && !mbar_wait(&bar.wempty[ws], ((wi / WS) - 1) & 1)) { ok = false; break; }
              const int wrow = (q * NK + k) * Gm::WROWS + b * Gm::MMA_N;
              if (issuer) mbar_arrive_expect_tx(&bar.wfull[ws], (uint32_t)Gm::W_BOX);  // (pairs) both halves
              if (P2)  // this CTA's half of the box's rows
                tma_load_2d_pair(wring + ws * Cf::WB, &tmWh, dsmem_addr(&bar.wfull[ws], 0), 0,
                                 wrow + prk * (Gm::MMA_N / 2));
              else
                tma_load_2d(wring + ws * Cf::WB, &tmW, &bar.wfull[ws], 0, wrow);
              ++wi;
            }
          }
        }
      }
      if (!ok) {
        raise_error(err, ERR_TIMEOUT);
        bar.abort_flag = 1;
      }
      // Drain: every copy started here has landed before the CTA can leave.  (Pairs: the
      // copies count on the even CTA's barriers; the MMAs' release of each slot, which
      // arrives on this CTA's barriers, follows them, and no arrival is left in flight.)
      for (uint32_t i = xi > (uint32_t)XS ? xi - XS : 0; i < xi; ++i)
        if (!mbar_wait(P2 ? &bar.xempty[i % XS] : &bar.xfull[i % XS], (i / XS) & 1)) raise_error(err, ERR_TIMEOUT);
      for (uint32_t i = wi > (uint32_t)WS ? wi - WS : 0; i < wi; ++i)
        if (!mbar_wait(P2 ? &bar.wempty[i % WS] : &bar.wfull[i % WS], (i / WS) & 1)) raise_error(err, ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && issuer) {
      // ---------------- MMA issuer (pairs: the even CTA, M = 256 over both CTAs' tokens)
      constexpr uint32_t idesc = idesc_bf16_f32(P2 ? 2 * RT_BM : RT_BM, Gm::MMA_N);
      uint32_t xi = 0, wi = 0;
      int lt = 0;
      bool ok = true;
      for (int it = it0; it < n_items && ok; it += istep, ++lt) {
        if (bar.abort_flag) { ok = false; break; }
        const int buf = lt % NBUF;
        if (lt >= NBUF && !mbar_wait(&bar.aempty[buf], ((lt / NBUF) - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(buf * Gm::TILE_COLS);
        for (int xs = 0; xs < NXS && ok; ++xs) {
          const int slot = (int)(xi % XS);
          if (!mbar_wait(&bar.xfull[slot], (xi / XS) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t xa0 = smem_u32(xring + slot * Cf::X_STAGE);
          for (int at = 0; at < NAX && ok; ++at) {
            const int k = xs * NAX + at;
            if (k >= NK) break;
            const uint32_t xa = xa0 + at * Cf::X_ATOM;
#pragma unroll
            for (int b = 0; b < Gm::WBOXES; ++b) {
              const int ws = (int)(wi % WS);
              if (!mbar_wait(&bar.wfull[ws], (wi / WS) & 1)) { ok = false; break; }
              tc_fence_after();
              const uint32_t wa = smem_u32(wring + ws * Cf::WB);
#pragma unroll
              for (int kk = 0; kk < RT_BK / 16; ++kk) {
                const bool first = k == 0 && kk == 0 && !(EC == 256 && (ONE ? b > 0 : b == 2));
                if (P2)
                  tc_mma_bf16_pair(acc + Gm::dcol(b), sw128_kmajor_desc(xa + kk * 32),
                                   sw128_kmajor_desc(wa + kk * 32), idesc, first ? 0u : 1u);
                else
                  tc_mma_bf16(acc + Gm::dcol(b), sw128_kmajor_desc(xa + kk * 32), sw128_kmajor_desc(wa + kk * 32),
                              idesc, first ? 0u : 1u);
              }
              if (P2)
                tc_commit_pair(&bar.wempty[ws], (uint16_t)3u);
              else
                tc_commit(&bar.wempty[ws]);
              ++wi;
            }
          }
          if (P2)
            tc_commit_pair(&bar.xempty[slot], (uint16_t)3u);
          else
            tc_commit(&bar.xempty[slot]);
          ++xi;
        }
        if (P2)
          tc_commit_pair(&bar.afull[buf], (uint16_t)3u);
        else
          tc_commit(&bar.afull[buf]);  // arrives once every MMA of the tile has completed
      }
      if (!ok) {
        raise_error(err, ERR_TIMEOUT);
        bar.abort_flag = 1;
      }
      // every MMA issued above has completed before TMEM can be freed
      if (P2)
        tc_commit_pair(&bar.drain, (uint16_t)1u);
      else
        tc_commit(&bar.drain);
      if (!mbar_wait(&bar.drain, 0)) raise_error(err, ERR_TIMEOUT);
      // (pairs) the last items' releases from the odd CTA have arrived before this CTA leaves
      if (P2 && ok)
        for (int i = lt > NBUF ? lt - NBUF : 0; i < lt; ++i)
          if (!mbar_wait(&bar.aempty[i % NBUF], (i / NBUF) & 1)) raise_error(err, ERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2 .. 17)
    // Warp w reads TMEM lane quadrant lq = w % 4 (tokens 32 lq .. 32 lq + 31) and column
    // group cg = (w - 2) / 4 (CPW consecutive experts); NCG groups cover the CTA's EC experts.
    constexpr int NCG = EC >= 64 ? 4 : EC / 16;
    constexpr int CPW = EC / NCG;
    const int lq = warp & 3, cg = (warp - 2) >> 2;
    const bool has_cols = cg < NCG;
    const int cbeg = cg * CPW;
    const int i = lq * 32 + lane;
    const int et = threadIdx.x - 64;  // 0 .. 511
    const bool leader = et == 0;
    int lt = 0;
    for (int it = it0; it < n_items; it += istep, ++lt) {
      const int buf = lt % NBUF;
      const int q = GX ? it % Q : qc;
      const int tid = P2 ? 2 * (it / Q) + prk : GX ? it / Q : it;
      const int e0 = q * EC;
      const int g = tid / nT, tile = tid - g * nT;
      const int t0 = tile * RT_BM;
      const long long tok0 = (long long)g * T + t0;
      const bool valid = t0 + i < T;
      const long long tok = tok0 + i;
      const uint32_t trow = tmem + (uint32_t)(buf * Gm::TILE_COLS) + ((uint32_t)(lq * 32) << 16);
      if (GX)  // this item's slice of the bias (the previous item's epilogue is done with it)
        for (int c = et; c < EC; c += 32 * RT_EPI_WARPS)
          sh.bias[c] = e0 + c < E ? (br ? br[e0 + c] : 0.f) : -INFINITY;

      if (leader) {  // the tile's accumulator is complete (or the kernel is giving up)
        int ok = bar.abort_flag ? 0 : 1;
        if (ok && !mbar_wait(&bar.afull[buf], (lt / NBUF) & 1)) {
          raise_error(err, ERR_TIMEOUT);
          ok = 0;
        }
        if (!ok) bar.abort_flag = 1;
        bar.ep_ok = ok;
      }
      rt_epi_sync();
      if (!bar.ep_ok) break;
      tc_fence_after();
      if (P2 && tid >= total_tiles) {  // the pair's second tile past the last one: release only
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(&bar.aempty[buf], 0u);
        rt_epi_sync();  // every thread has read ep_ok before the leader writes it again
        continue;
      }

      // pass 1: logits z (+ bias) into registers; max / argmax over this warp's columns
      // (increasing e with strict >, so the lowest index wins a tie)
      float v[CPW];
      float m = -INFINITY, m2 = -INFINITY;  // (T2) m2, a2: the second-highest logit and its expert
      int a = INT_MAX, a2 = INT_MAX;
      if (has_cols) {
#pragma unroll
        for (int ch = 0; ch < CPW / 8; ++ch) {
          const uint32_t col = (uint32_t)(cbeg + ch * 8);
          uint32_t h[8], r1[8], r2[8];
          if (Gm::ACC_BLOCKS == 1 && (ch & 3) == 0) {  // four chunks' loads before one wait
            uint32_t h1[8], h2[8], h3[8];
            tmem_ld8(trow + col, h);
            tmem_ld8(trow + col + 8, h1);
            tmem_ld8(trow + col + 16, h2);
            tmem_ld8(trow + col + 24, h3);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              v[ch * 8 + 8 + j] = __uint_as_float(h1[j]);
              v[ch * 8 + 16 + j] = __uint_as_float(h2[j]);
              v[ch * 8 + 24 + j] = __uint_as_float(h3[j]);
              r1[j] = 0u;
            }
          } else if (Gm::ACC_BLOCKS == 1) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              h[j] = __float_as_uint(v[ch * 8 + j]);
              r1[j] = 0u;
            }
          } else if (Gm::ACC_BLOCKS == 2 && (ch & 1) == 0) {  // two chunks' loads before one wait
            uint32_t h2[8], q2[8];
            tmem_ld8(trow + col, h);
            tmem_ld8(trow + EC + col, r1);
            tmem_ld8(trow + col + 8, h2);
            tmem_ld8(trow + EC + col + 8, q2);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              v[ch * 8 + 8 + j] = __uint_as_float(h2[j]) + __uint_as_float(q2[j]);
            }
          } else if (Gm::ACC_BLOCKS == 2) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              h[j] = __float_as_uint(v[ch * 8 + j]);
              r1[j] = 0u;
            }
          } else {
            tmem_ld8(trow + col, h);
            tmem_ld8(trow + EC + col, r1);
            if (Gm::ACC_BLOCKS == 3) tmem_ld8(trow + 2 * EC + col, r2);
            tmem_ld_wait();
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = cbeg + ch * 8 + j;
            const float corr = Gm::ACC_BLOCKS == 3   ? __uint_as_float(r1[j]) + __uint_as_float(r2[j])
                               : Gm::ACC_BLOCKS == 2 ? __uint_as_float(r1[j])
                                                     : 0.f;
            const float z = (__uint_as_float(h[j]) + corr) + sh.bias[c];
            v[ch * 8 + j] = z;
            if (z > m) {  // padding experts: z = -inf
              if (T2) { m2 = m; a2 = a; }
              m = z;
              a = e0 + c;
            } else if (T2 && z > m2) {
              m2 = z;
              a2 = e0 + c;
            }
          }
          if (logits && valid) {  // the chunk's 8 logits of this token: 16-byte stores when aligned
            const int c0 = e0 + cbeg + ch * 8;
            float* dst = logits + tok * E + c0;
            if ((E & 3) == 0 && c0 + 8 <= E) {
#pragma unroll
              for (int q4 = 0; q4 < 2; ++q4)
                *reinterpret_cast<float4*>(dst + 4 * q4) =
                    make_float4(v[ch * 8 + 4 * q4], v[ch * 8 + 4 * q4 + 1], v[ch * 8 + 4 * q4 + 2],
                                v[ch * 8 + 4 * q4 + 3]);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (c0 + j < E) dst[j] = v[ch * 8 + j];
            }
          }
        }
      }
      // the accumulator set is read: the next tile's MMAs may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (P2)  // on the even CTA's barrier (its own arrival is local)
          mbar_arrive_remote(&bar.aempty[buf], 0u);
        else
          mbar_arrive(&bar.aempty[buf]);
      }

      if (has_cols) {
        sh.red_m[cg][i] = m;
        sh.red_a[cg][i] = a;
        if (T2) {
          sh.red_m2[cg][i] = m2;
          sh.red_a2[cg][i] = a2;
        }
      }
      rt_epi_sync();
      float mc = -INFINITY, mc2 = -INFINITY;  // max (and, T2, second) over this CTA's experts
      int ac = INT_MAX, ac2 = INT_MAX;
#pragma unroll
      for (int k = 0; k < NCG; ++k) {
        if (T2)
          top2_merge(mc, ac, mc2, ac2, sh.red_m[k][i], sh.red_a[k][i], sh.red_m2[k][i], sh.red_a2[k][i]);
        else if (sh.red_m[k][i] > mc) {
          mc = sh.red_m[k][i];
          ac = sh.red_a[k][i];
        }
      }

      // pass 1b: exp(z - mc) in registers, partial sums
      float ps = 0.f;
      if (has_cols) {
        const float mcs = mc * LOG2E;
#pragma unroll
        for (int k = 0; k < CPW; ++k) {
          const float ex = ex2_approx(fmaf(v[k], LOG2E, -mcs));  // 0 for padding experts (z = -inf)
          v[k] = ex;
          ps += ex;
        }
        sh.red_s[cg][i] = ps;
      }
      if (!GX && Q > 1 && leader) {
        int ok = 1;
        // every peer has read its receive buffer of the previous tile
        if (lt >= 1 && !mbar_wait_cluster(&bar.rfree, (lt - 1) & 1)) {
          raise_error(err, ERR_TIMEOUT);
          bar.abort_flag = 1;
          ok = 0;
        }
        // arm this CTA's receive barrier for the tile: Q slices of 12 (T2: 20) bytes per token
        mbar_arrive_expect_tx(&bar.rfull, (uint32_t)(Q * RT_BM * (T2 ? 20 : 12)));
        bar.ep_ok = ok;
      }
      rt_epi_sync();
      const size_t xrow = (size_t)tid * Q;  // (global) the tile's exchange rows
      if (cg == 0) {
        float sc = 0.f;
#pragma unroll
        for (int k = 0; k < NCG; ++k) sc += sh.red_s[k][i];
        if (GX) {
          xms[(xrow + q) * RT_BM + i] = make_float2(mc, sc);
          xam[(xrow + q) * RT_BM + i] = ac;
          if (T2) {
            xm2[(xrow + q) * RT_BM + i] = mc2;
            xa2[(xrow + q) * RT_BM + i] = ac2;
          }
        } else if (Q > 1) {  // into slot q of every peer's receive buffer
          for (int rk = 0; rk < Q; ++rk) {
            st_async_v2_f32(&sh.rms[q][i], mc, sc, &bar.rfull, (uint32_t)rk);
            st_async_s32(&sh.ra[q][i], ac, &bar.rfull, (uint32_t)rk);
            if (T2) {
              st_async_s32(&sh.rm2[q][i], __float_as_int(mc2), &bar.rfull, (uint32_t)rk);
              st_async_s32(&sh.ra2[q][i], ac2, &bar.rfull, (uint32_t)rk);
            }
          }
        } else {
          sh.rms[0][i] = make_float2(mc, sc);
          sh.ra[0][i] = ac;
          if (T2) {
            sh.rm2[0][i] = __float_as_int(mc2);
            sh.ra2[0][i] = ac2;
          }
        }
      }
      bool xok = true;
      if (GX) {
        rt_epi_sync();  // this slice's 128 rows are written
        if (warp == 2) {  // the leader's warp: publish, then lane k watches slice k's flag
          bool ok = bar.abort_flag == 0;
          if (leader) {
            __threadfence();
            st_release_gpu(xflag + xrow + q, epoch);
          }
          __syncwarp();
          const long long t0 = clock64();
          bool seen = lane >= Q;
          while (ok) {
            if (!seen) seen = ld_acquire_gpu(xflag + xrow + lane) == epoch;
            if (__all_sync(0xffffffffu, seen)) break;
            if (__shfl_sync(0xffffffffu, clock64() - t0 > WAIT_LIMIT_CYCLES ? 1 : 0, 0)) {
              if (leader) {
                raise_error(err, ERR_TIMEOUT);
                bar.abort_flag = 1;
              }
              ok = false;
            }
          }
          if (leader) bar.ep_ok = ok ? 1 : 0;
        }
        rt_epi_sync();
        xok = bar.ep_ok != 0;
      } else if (Q > 1) {
        if (leader) {
          int ok = bar.ep_ok;
          if (ok && !mbar_wait_cluster(&bar.rfull, lt & 1)) {
            raise_error(err, ERR_TIMEOUT);
            bar.abort_flag = 1;
            ok = 0;
          }
          bar.ep_ok = ok;
        }
        rt_epi_sync();
        xok = bar.ep_ok != 0;
      } else {
        rt_epi_sync();
      }
      if (cg == 0) {
        float M = -INFINITY, S = 0.f, M2 = -INFINITY;
        int A = INT_MAX, A2 = INT_MAX;
        if (xok && GX) {  // expert slices in order: the lowest index wins a tie
          float2 ms[8];  // every slice's pair in flight at once (Q <= 8)
#pragma unroll
          for (int rk = 0; rk < 8; ++rk)
            if (rk < Q) ms[rk] = __ldcg(xms + (xrow + rk) * RT_BM + i);
          int kb = 0;
#pragma unroll
          for (int rk = 0; rk < 8; ++rk)
            if (rk < Q && ms[rk].x > M) {
              M = ms[rk].x;
              kb = rk;
            }
          if (M > -INFINITY) A = __ldcg(xam + (xrow + kb) * RT_BM + i);
#pragma unroll
          for (int rk = 0; rk < 8; ++rk)
            if (rk < Q && ms[rk].y > 0.f) S += ms[rk].y * expf(ms[rk].x - M);
          if (T2) {  // second: the best slice's own second, or the best first of another slice
            float Mo = -INFINITY;
            int ko = -1;
#pragma unroll
            for (int rk = 0; rk < 8; ++rk)
              if (rk < Q && rk != kb && ms[rk].x > Mo) {
                Mo = ms[rk].x;
                ko = rk;
              }
            const float mk2 = __ldcg(xm2 + (xrow + kb) * RT_BM + i);
            // on a tie the lower expert index wins: slice ko's experts rank before kb's when ko < kb
            const bool other = ko >= 0 && (Mo > mk2 || (Mo == mk2 && ko < kb));
            M2 = other ? Mo : mk2;
            A2 = other ? __ldcg(xam + (xrow + ko) * RT_BM + i) : __ldcg(xa2 + (xrow + kb) * RT_BM + i);
          }
        } else if (xok) {  // expert slices in rank order: the lowest index wins a tie
          for (int rk = 0; rk < Q; ++rk) {
            const float mr = sh.rms[rk][i].x;
            if (T2) {
              top2_merge(M, A, M2, A2, mr, sh.ra[rk][i], __int_as_float(sh.rm2[rk][i]), sh.ra2[rk][i]);
            } else if (mr > M) {
              M = mr;
              A = sh.ra[rk][i];
            }
          }
          for (int rk = 0; rk < Q; ++rk) {
            const float2 ms = sh.rms[rk][i];
            if (ms.y > 0.f) S += ms.y * expf(ms.x - M);
          }
        }
        if (A < 0 || A >= E) {  // only non-finite logits (or a failed exchange) get here
          if (valid) raise_error(err, ERR_BOUNDS);
          A = 0;
        }
        if (T2) {
          if (A2 < 0 || A2 >= E || A2 == A) {  // the same (E >= 2)
            if (valid) raise_error(err, ERR_BOUNDS);
            A2 = A == 0 ? 1 : 0;
          }
          sh.M2all[i] = M2;
          sh.texp2[i] = valid ? A2 : -1;
        }
        sh.Mall[i] = M;
        sh.Sall[i] = S;
        sh.texp[i] = valid ? A : -1;
        const float lse = M + logf(S);  // log sum_e exp z_e over all E experts (router z-loss)
        sh.zz[i] = valid ? lse * lse : 0.f;
      }
      rt_epi_sync();
      // this CTA has read its receive buffer (every read value was consumed before the
      // barrier above): peers may fill it with the next tile
      if (!GX && Q > 1 && leader)
        for (int rk = 0; rk < Q; ++rk) mbar_arrive_remote_relaxed(&bar.rfree, (uint32_t)rk);

      // pass 2: p = exp(z - mc) * exp(mc - M) / S; column sums over the tile's tokens
      const float scale = valid ? expf(mc - sh.Mall[i]) / sh.Sall[i] : 0.f;
      if (has_cols) {
#pragma unroll
        for (int ch = 0; ch < CPW / 8; ++ch) {
          float* p = v + ch * 8;  // scaled in place: exp(z - mc) is not needed afterwards
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = cbeg + ch * 8 + j;
            p[j] *= scale;  // 0 past E (v = 0) and for invalid tokens (scale = 0)
            if (probs && valid && e0 + c < E) probs[tok * E + e0 + c] = p[j];
          }
          const float cs = warp_colsum8(p, lane);
          if ((lane & 3) == 0) sh.colsum[lq][cbeg + ch * 8 + (lane >> 2)] = cs;
        }
      }
      const int A = sh.texp[i];
      if (cg == 0 && A >= e0 && A < e0 + EC) atomicAdd(&sh.hist[A - e0], 1);
      if (T2) {
        const int A2 = sh.texp2[i];
        if (cg == 0 && A2 >= e0 && A2 < e0 + EC) atomicAdd(&sh.hist2[A2 - e0], 1);
      }
      rt_epi_sync();

      const size_t tbase = ((size_t)g * nT + tile) * E;
      if (q == 0 && warp == 2) {  // the tile's sum of (log sum exp z)^2, fixed order
        float zs = (sh.zz[lane] + sh.zz[lane + 32]) + (sh.zz[lane + 64] + sh.zz[lane + 96]);
        zs = warp_sum(zs);
        if (lane == 0) tile_Z[(size_t)g * nT + tile] = zs;
      }
      for (int c = et; c < EC; c += 32 * RT_EPI_WARPS) {
        const int e = e0 + c;
        if (e < E) {
          tile_P[tbase + e] = ((sh.colsum[0][c] + sh.colsum[1][c]) + sh.colsum[2][c]) + sh.colsum[3][c];
          tile_hist[tbase + e] = sh.hist[c];
          if (T2) tile_hist2[tbase + e] = sh.hist2[c];
        }
        sh.hist[c] = 0;  // for the next tile
        if (T2) sh.hist2[c] = 0;
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
        if (T2) {  // the second choice: its rank among the tile's second choices; the pair's softmax
          const int A2 = sh.texp2[i];
          const int key2 = valid ? A2 : -1 - lane;
          const unsigned same2 = __match_any_sync(0xffffffffu, key2);
          int rk2 = __popc(same2 & ((1u << lane) - 1u));
          for (int j = 0; j < lq * 32; ++j) rk2 += sh.texp2[j] == A2;
          if (valid) {
            const float u = expf(sh.M2all[i] - sh.Mall[i]);
            gate[tok] = 1.0f / (1.0f + u);
            gate2[tok] = u / (1.0f + u);
            expert2[tok] = A2;
            rank2[tok] = rk2;
          }
        }
      }
      rt_epi_sync();  // the tile's scratch is read before the next tile writes it
    }
  }

  tc_fence_before();
  __syncthreads();
  if ((!GX && Q > 1) || P2) cluster_sync();  // no peer reads this CTA's shared memory or arrives on its barriers any more
  if (GX && threadIdx.x == 0) {  // the last CTA to finish advances the epoch for the next launch
    __threadfence();
    if (atomicAdd(xctl + 1, 1u) == gridDim.x - 1) {
      xctl[1] = 0u;
      __threadfence();
      st_release_gpu(xctl, epoch);
    }
  }
  if (warp == 1) {
    if (P2)
      tmem_dealloc_pair(tmem, Gm::TMEM_COLS);
    else
      tmem_dealloc(tmem, Gm::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
// CTAs of router_tc_kernel<EC, NAX, XM> resident at once in clusters of cl CTAs (cached per
// kernel, device and cluster size).
template <int EC, int NAX, int XM, bool T2 = false, bool ONE = false>
static int rt_fit(int cl) {
  static std::atomic<int> cache[64][9];  // handles on several host threads may fill it
  auto kern = router_tc_kernel<EC, NAX, XM, T2, ONE>;
  constexpr int smem = rt_smem_bytes<EC, NAX, XM == 2, T2>();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const bool cached = dev >= 0 && dev < 64 && cl >= 1 && cl <= 8;
  if (cached) {
    const int c = cache[dev][cl].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cl > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cl, 1, 1);
    cfg.blockDim = dim3(RT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)cl;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = device_sm_count() / cl;
    }
    n *= cl;
  } else {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, RT_THREADS, (size_t)smem) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 1;
    }
    n *= device_sm_count();
  }
  if (n < cl) n = cl;
  if (cached) cache[dev][cl].store(n, std::memory_order_relaxed);
  return n;
}

// Exchange rows of the global variant for `tiles` token tiles: (max, sum) float2 and argmax
// int per (tile, slice, token), a flag per (tile, slice), then the epoch and ticket words.
struct RtXchg {
  float2* ms;
  int* am;
  uint32_t* flag;
  uint32_t* ctl;
  float* m2;  // (top-2) each slice's second logit and expert per token
  int* a2;
};
static size_t rt_round256(size_t b) { return (b + 255) / 256 * 256; }
static bool rt_global(int E) {
  const int EC = router_tc_experts_per_cta(E);
  return (E + EC - 1) / EC > 2;
}
bool router_tc_top2_fused(int E, int d) {
  return E >= 2 && d % (2 * RT_BK) == 0;
}

size_t router_tc_exchange_bytes(long long tiles, int E, bool top2) {
  if (!rt_global(E) || tiles <= 0) return 0;
  const int EC = router_tc_experts_per_cta(E);
  const size_t n = (size_t)tiles * (size_t)((E + EC - 1) / EC);
  return rt_round256(n * RT_BM * sizeof(float2)) + rt_round256(n * RT_BM * sizeof(int)) +
         rt_round256(n * sizeof(uint32_t)) + 256 +
         (top2 ? rt_round256(n * RT_BM * sizeof(float)) + rt_round256(n * RT_BM * sizeof(int)) : 0);
}
static RtXchg rt_xchg(void* base, long long tiles, int Q) {
  uint8_t* p = static_cast<uint8_t*>(base);
  const size_t n = (size_t)tiles * Q;
  RtXchg x;
  x.ms = reinterpret_cast<float2*>(p);
  p += rt_round256(n * RT_BM * sizeof(float2));
  x.am = reinterpret_cast<int*>(p);
  p += rt_round256(n * RT_BM * sizeof(int));
  x.flag = reinterpret_cast<uint32_t*>(p);
  p += rt_round256(n * sizeof(uint32_t));
  x.ctl = reinterpret_cast<uint32_t*>(p);
  p += 256;
  x.m2 = reinterpret_cast<float*>(p);  // present only in buffers sized for top-2
  p += rt_round256(n * RT_BM * sizeof(float));
  x.a2 = reinterpret_cast<int*>(p);
  return x;
}

template <int EC, int NAX, int XM, bool T2 = false, bool ONE = false>
static cudaError_t rt_launch(int grid, int cluster, bool coop, bool pdl, cudaStream_t s, const CUtensorMap& tmX,
                             const CUtensorMap& tmW, const CUtensorMap& tmWh, const RouteArgs& a, int nT, int Q,
                             int total, int32_t* rank, const RtXchg& x) {
  auto kern = router_tc_kernel<EC, NAX, XM, T2, ONE>;
  constexpr int smem = rt_smem_bytes<EC, NAX, XM == 2, T2>();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(RT_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[3];
  unsigned n = 0;
  if (coop) {  // the CTAs wait on one another's exchange flags: all must be resident
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, tmX, tmW, tmWh, a.br, a.T, a.E, a.d, nT, Q, total, a.expert, a.gate, rank,
                            a.tile_hist, a.tile_P, a.tile_Z, a.logits_out, a.probs, a.err, x.ms, x.am, x.flag, x.ctl,
                            T2 ? a.expert2 : nullptr, T2 ? a.gate2 : nullptr, T2 ? a.slot2 : nullptr,
                            T2 ? a.tile_hist2 : nullptr, T2 && XM >= 1 ? x.m2 : nullptr,
                            T2 && XM >= 1 ? x.a2 : nullptr);
}

// Widest d for which 256-expert slices sum all three pieces in one accumulator block (RtGeom).
constexpr int RT_ONE_ACC_MAX_D = 1024;

// CTA pairs need a cooperative launch of 2-CTA clusters; a device that refuses it gets the
// one-CTA global variant from then on.
static std::atomic<bool> g_rt_pair_refused[64];

// CTAs resident at once, lowered to the caller's budget (> 0) but never below the fewest
// that keep every wait of the kernel on running work (need: one cluster of Q; one CTA per
// slice of a tile for the global exchange; a pair per slice for CTA pairs).
static int rt_budget(int fit, int max_ctas, int need) {
  if (max_ctas <= 0 || max_ctas >= fit) return fit;
  return max_ctas > need ? max_ctas : (need < fit ? need : fit);
}

template <int EC, int NAX>
static int launch_rt(const CUtensorMap& tmX, const CUtensorMap& tmW, const CUtensorMap& tmWh, const RouteArgs& a,
                     int nT, int Q, int32_t* rank, cudaStream_t s) {
  const long long total = (long long)a.G * nT;
  if (total * Q >= (1ll << 31)) return -1;
  if (a.xchg && rt_global(a.E)) {
    const RtXchg x = rt_xchg(a.xchg, total, Q);
    if (a.top2) {  // top-2 in the router: slices of 64 to 256 (256: CTA pairs when they run)
      if constexpr ((EC == 64 || EC == 128 || EC == 256) && NAX == 2) {
        const long long items = total * Q;
        if constexpr (EC == 256) {
          int dev = 0;
          if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
          if (a.max_ctas == 0 && total >= 2 &&
              !(dev >= 0 && dev < 64 && g_rt_pair_refused[dev].load(std::memory_order_relaxed))) {
            const bool one = a.d <= RT_ONE_ACC_MAX_D;
            const long long pitems = (total + 1) / 2 * Q;
            const int pfit = (one ? rt_fit<EC, NAX, 2, true, true>(2) : rt_fit<EC, NAX, 2, true>(2)) / 2;
            const int pairs = (int)(pitems < pfit ? pitems : pfit);
            if ((one ? rt_launch<EC, NAX, 2, true, true>(2 * pairs, 2, true, false, s, tmX, tmW, tmWh, a, nT, Q,
                                                         (int)total, rank, x)
                     : rt_launch<EC, NAX, 2, true>(2 * pairs, 2, true, false, s, tmX, tmW, tmWh, a, nT, Q,
                                                   (int)total, rank, x)) == cudaSuccess)
              return 1;
            cudaGetLastError();
            if (dev >= 0 && dev < 64) g_rt_pair_refused[dev].store(true, std::memory_order_relaxed);
          }
          if (a.d <= RT_ONE_ACC_MAX_D) {
            const int fit = rt_budget(rt_fit<EC, NAX, 1, true, true>(1), a.max_ctas, Q);
            const int grid = (int)(items < fit ? items : fit);
            return rt_launch<EC, NAX, 1, true, true>(grid, 1, true, false, s, tmX, tmW, tmWh, a, nT, Q, (int)total,
                                                     rank, x) == cudaSuccess
                       ? 1
                       : -1;
          }
        }
        const int fit = rt_budget(rt_fit<EC, NAX, 1, true>(1), a.max_ctas, Q);
        const int grid = (int)(items < fit ? items : fit);
        return rt_launch<EC, NAX, 1, true>(grid, 1, true, false, s, tmX, tmW, tmWh, a, nT, Q, (int)total, rank,
                                           x) == cudaSuccess
                   ? 1
                   : -1;
      }
      return -1;
    }
    if constexpr (EC == 256) {
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
      // (with a CTA budget: single CTAs, which fit on SMs that another kernel frees one at a time)
      if (a.max_ctas == 0 && total >= 2 &&
          !(dev >= 0 && dev < 64 && g_rt_pair_refused[dev].load(std::memory_order_relaxed))) {
        const long long pitems = (total + 1) / 2 * Q;
        const int fit = rt_budget(a.d <= RT_ONE_ACC_MAX_D ? rt_fit<EC, NAX, 2, false, true>(2) : rt_fit<EC, NAX, 2>(2),
                                  a.max_ctas, 2 * Q) /
                        2;
        const int pairs = (int)(pitems < fit ? pitems : fit);
        if ((a.d <= RT_ONE_ACC_MAX_D
                 ? rt_launch<EC, NAX, 2, false, true>(2 * pairs, 2, true, false, s, tmX, tmW, tmWh, a, nT, Q,
                                                      (int)total, rank, x)
                 : rt_launch<EC, NAX, 2>(2 * pairs, 2, true, false, s, tmX, tmW, tmWh, a, nT, Q, (int)total, rank,
                                         x)) == cudaSuccess)
          return 1;
        cudaGetLastError();
        if (dev >= 0 && dev < 64) g_rt_pair_refused[dev].store(true, std::memory_order_relaxed);
      }
    }
    const long long items = total * Q;
    if constexpr (EC == 256) {
      if (a.d <= RT_ONE_ACC_MAX_D) {
        const int fit = rt_budget(rt_fit<EC, NAX, 1, false, true>(1), a.max_ctas, Q);
        const int grid = (int)(items < fit ? items : fit);
        return rt_launch<EC, NAX, 1, false, true>(grid, 1, true, false, s, tmX, tmW, tmWh, a, nT, Q, (int)total,
                                                  rank, x) == cudaSuccess
                   ? 1
                   : -1;
      }
    }
    const int fit = rt_budget(rt_fit<EC, NAX, 1>(1), a.max_ctas, Q);
    const int grid = (int)(items < fit ? items : fit);
    return rt_launch<EC, NAX, 1>(grid, 1, true, false, s, tmX, tmW, tmWh, a, nT, Q, (int)total, rank, x) ==
                   cudaSuccess
               ? 1
               : -1;
  }
  if (a.top2) {  // top-2 routing in the router (slices of at most 64 experts meeting in a cluster)
    if constexpr (EC <= 64 && NAX == 2) {
      const int fit = rt_budget(rt_fit<EC, NAX, 0, true>(Q), a.max_ctas, Q) / Q;
      const int ncl = (int)(total < fit ? total : fit);
      return rt_launch<EC, NAX, 0, true>(Q * ncl, Q, false, true, s, tmX, tmW, tmWh, a, nT, Q, (int)total, rank,
                                         RtXchg{}) == cudaSuccess
                 ? 1
                 : -1;
    }
    return -1;
  }
  const int fit = rt_budget(rt_fit<EC, NAX, 0>(Q), a.max_ctas, Q) / Q;
  const int ncl = (int)(total < fit ? total : fit);
  return rt_launch<EC, NAX, 0>(Q * ncl, Q, false, true, s, tmX, tmW, tmWh, a, nT, Q, (int)total, rank, RtXchg{}) ==
                 cudaSuccess
             ? 1
             : -1;
}

// Experts per CTA: the smallest power of two >= 16 that keeps the cluster at <= 8
// CTAs, raised to 64 when E allows (fewer CTAs re-reading each token tile).
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
  const size_t NK = (size_t)((d + RT_BK - 1) / RT_BK);
  return Q * EC * 3 * NK * RT_BK * 2;
}

int launch_router_split(const float* Wr, void* wsplit, int E, int d, cudaStream_t s) {
  const int EC = router_tc_experts_per_cta(E);
  const int Q = (E + EC - 1) / EC;
  const int NK = (d + RT_BK - 1) / RT_BK;
  const long long n = (long long)Q * EC * NK * RT_BK;
  const unsigned sb = (unsigned)((n + 255) / 256 < 148 * 16 ? (n + 255) / 256 : 148 * 16);
  return launch_k(router_split_kernel, dim3(sb), dim3(256), 0, s, false, 1, Wr, (__nv_bfloat16*)wsplit, E, d, EC, NK,
                  n) == cudaSuccess
             ? 1
             : -1;
}

int launch_router_tc(const RouteArgs& a, int32_t* rank, cudaStream_t s) {
  const long long N = (long long)a.G * a.T;
  if (N == 0) return 0;
  const int nT = (a.T + RT_BM - 1) / RT_BM;
  const int EC = router_tc_experts_per_cta(a.E);
  const int Q = (a.E + EC - 1) / EC;
  if (EC > 256 || Q > 8) return -1;
  const int NK = (a.d + RT_BK - 1) / RT_BK;
  if ((long long)Q * NK * 3 * EC >= (1ll << 31)) return -1;  // TMA row coordinates are 32-bit
  int launches = 0;
  if (a.Wr) {  // else: the pieces prepared by an earlier split are used as they are
    if (launch_router_split(a.Wr, a.wsplit, a.E, a.d, s) < 0) return -1;
    ++launches;
  }
  const int nax = a.d % (2 * RT_BK) == 0 ? 2 : 1;  // x stages of two atoms (256 B per row) when d allows
  CUtensorMap tmX, tmW, tmWh;
  if (nax == 2) {
    if (!encode_bf16_3d(&tmX, a.x, (uint64_t)N, (uint64_t)a.d, RT_BM, 2u)) return -1;
  } else if (!encode_bf16_2d(&tmX, a.x, (uint64_t)N, (uint64_t)a.d, RT_BM)) {
    return -1;
  }
  if (!encode_bf16_2d(&tmW, a.wsplit, (uint64_t)3 * Q * EC * NK, (uint64_t)RT_BK, (uint32_t)router_tc_mma_n(EC)))
    return -1;
  tmWh = tmW;  // half boxes (CTA pairs split each W box's rows)
  if (EC == 256 && !encode_bf16_2d(&tmWh, a.wsplit, (uint64_t)3 * Q * EC * NK, (uint64_t)RT_BK, 128u)) return -1;
  int n2;
#define SMOE_RT(ECV) \
  n2 = nax == 2 ? launch_rt<ECV, 2>(tmX, tmW, tmWh, a, nT, Q, rank, s) : launch_rt<ECV, 1>(tmX, tmW, tmWh, a, nT, Q, rank, s)
  switch (EC) {
    case 16: SMOE_RT(16); break;
    case 32: SMOE_RT(32); break;
    case 64: SMOE_RT(64); break;
    case 128: SMOE_RT(128); break;
    default: SMOE_RT(256); break;
  }
#undef SMOE_RT
  return n2 < 0 ? -1 : launches + 1;
}

}  // namespace smoe
