// Expert FFN of the Switch layer on 5th-generation tensor cores (tcgen05, sm_103a).
//
// The expert FFN is d -> d_ff, ReLU, d_ff -> d with biases ("混合专家",
// world.lapla.si/zh/moe, section 专家里面是什么); bf16 operands with float32
// accumulation follow the bfloat16 expert computation of the Switch Transformers
// card (ai-papers.xuzou.cn, 方法适配), where only the router runs in float32.
// With the combine fused in, the second layer's epilogue writes
//     y_t = gate_t * FFN(x_t) (+ x_t)
// straight to token order ("042 · Switch Transformer：每个词只选一个专家", section 一;
// the gate is used as is, never renormalised).
//
// One persistent kernel runs both layers of every expert.  A tile is
//     out^T[m, n] = sum_k W[e, m, k] * in[e*R + n, k],  m in a 128-row block, n in a BN-row chunk
// ("swap AB": the expert's weight rows fill the 128-row MMA, its tokens are the N side).
// Layer-1 tiles (W1, input xe) write h; layer-2 tiles (W2, input h) write ye, or y
// when the combine is fused.  Tiles are handed out by an atomic ticket in an order
// that interleaves the layers: layer-1 tiles of expert s, then layer-2 tiles of
// expert s - LOOK (a lead of about 8 tiles per CTA), so h is read back from L2; a layer-2 tile waits
// (bounded) until all layer-1 tiles of its expert and chunk have been stored.
//
// Per CTA (one per SM, 64 + 256 MB threads):
//   warp 0, one lane : scheduler + TMA producer.  Takes tickets, publishes each tile in a
//                      small shared-memory queue, streams its W and activation tiles
//                      (128-byte swizzle) into a ring of stages (one barrier each).
//   warp 1, one lane : MMA issuer.  tcgen05.mma (M = 128 per weight block, N = BN, K = 16)
//                      into one of NBUF TMEM accumulator sets.
//   warps 2 ..       : epilogue, two warps per (weight block, TMEM lane quadrant), each
//                      taking alternate 32-column slices.  tcgen05.ld, + bias, ReLU
//                      (layer 1), bf16, store; layer 1 then publishes its chunk to the
//                      layer-2 tiles.
// Every wait is bounded; on timeout the CTA sets the error flag, stops taking tiles,
// drains its own copies and MMAs, frees TMEM and returns.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int FF_BM = 128;
constexpr int FF_BK = 64;          // 64 bf16 = 128 bytes = one swizzle atom
constexpr int FF_ATOM_A = FF_BM * FF_BK * 2;
// 64 + 256 MB threads: producer warp, MMA warp, 8 epilogue warps per 128-row weight block
constexpr int FF_EPW = 2;  // epilogue warps per (weight block, TMEM lane quadrant)
template <int MB> constexpr int ff_threads() { return 64 + 128 * FF_EPW * MB; }
constexpr int FF_SCHED = 4;        // tile queue depth
constexpr int FF_PB = 64;          // rows of the activation boxes used for partly filled chunks
constexpr int FF_MAX_STAGES = 8;
constexpr int FF_RING = 200 * 1024;

struct FfnParams {
  const __nv_bfloat16* b1;       // [E, F] or null
  const __nv_bfloat16* b2;       // [E, d] or null
  __nv_bfloat16* h;              // [E * R, F]
  __nv_bfloat16* out;            // ye [E * R, d], or y [N, d] with the combine
  const int32_t* expert_rows;    // [E]
  const int32_t* tok_of_row;     // [E * R] (combine)
  const float* gate;             // [N] (combine)
  const __nv_bfloat16* resid;    // [N, d] or null (combine)
  const __nv_bfloat16* hmask;    // [E * R, F]: with MASK, layer 1 keeps its sum where this is > 0
  uint32_t* next_tile;           // zero at launch
  uint32_t* done1;               // [E * NCH], zero at launch
  uint32_t* done2;               // [E * NCH], zero at launch: layer-2 tiles of (expert, chunk) done
  uint32_t* err;
  int E, R, d, F, BN, NCH, LOOK, NA, STAGES, stage_bytes, combine, w_evict_first;
  int MB;                        // 128-row weight blocks per tile (the kernel's template value)
  int layer2;                    // 0: layer-1 tiles only (a weight gradient)
  int stall;                     // test only: tile (layer 1, expert 0, block 0, chunk 0) never publishes
  int discard_h;                 // h is scratch: the last layer-2 tile of a chunk drops its lines from L2
  float* out_f32;                // MODE 2: the float32 result [E * R, F] (R: tokens, F: features)
  const int32_t* kcount;         // MODE 2 (or null): rows of expert e on the contraction axis; only
                                 // their 64-row atoms are read (at least one, zero past the count)
};

struct FfTile {
  int layer, e, mt, nc;
};

// Ticket -> tile.  Per expert: S1 = NCH * F/(128 MB) layer-1 tiles, S2 = NCH * d/(128 MB)
// layer-2 tiles (m-block major, chunk minor).  Order: layer 1 of experts 0..L-1; then, for
// s = L..E-1, layer 1 of s followed by layer 2 of s - L; then layer 2 of the last L.
// Returns false past the last tile.
__device__ __forceinline__ bool ff_decode(uint32_t t, const FfnParams& p, FfTile& tl) {
  const uint32_t S1 = (uint32_t)p.NCH * (uint32_t)(p.F / (FF_BM * p.MB));
  const uint32_t S2 = p.layer2 ? (uint32_t)p.NCH * (uint32_t)(p.d / (FF_BM * p.MB)) : 0u;
  const uint32_t L = (uint32_t)min(p.LOOK, p.E);
  const uint32_t E = (uint32_t)p.E;
  uint32_t r;
  if (t < L * S1) {
    tl.layer = 0;
    tl.e = (int)(t / S1);
    r = t % S1;
  } else if ((t -= L * S1) < (E - L) * (S1 + S2)) {
    const uint32_t step = L + t / (S1 + S2);
    r = t % (S1 + S2);
    if (r < S1) {
      tl.layer = 0;
      tl.e = (int)step;
    } else {
      tl.layer = 1;
      tl.e = (int)(step - L);
      r -= S1;
    }
  } else if ((t -= (E - L) * (S1 + S2)) < L * S2) {
    tl.layer = 1;
    tl.e = (int)(E - L + t / S2);
    r = t % S2;
  } else {
    return false;
  }
  tl.mt = (int)(r / (uint32_t)p.NCH);
  tl.nc = (int)(r % (uint32_t)p.NCH);
  return true;
}

struct FfShared {
  uint64_t full[FF_MAX_STAGES], empty[FF_MAX_STAGES];
  uint64_t sfull[FF_SCHED], sempty[FF_SCHED];
  uint64_t afull[2], aempty[2];
  int4 sched[FF_SCHED];
  int sched_nv[FF_SCHED];  // rows of the tile's token chunk that hold tokens (1 .. BN)
  int4 ep_tile;       // epilogue: the leader's tile, broadcast by a named barrier
  int ep_nv;
  // per epilogue warp: 16 tokens x 32 features (as 8 token pairs x 32 features, 32-bit
  // words), read back as 16-byte vectors
  alignas(16) __nv_bfloat16 xpose[8 * FF_EPW][16][32];
  int tok[256];       // combine: token of each column of the current layer-2 tile
  float gate[256];    // and its gate
  uint32_t tmem_slot;
  volatile int abort_flag;
  int ep_ok;
  int ep_acc_ok;
  int4 ep_disc;       // (flag, expert, first row, rows): the previous tile was the last reader of
                      // that chunk's h
};
static_assert(offsetof(FfShared, xpose) % 16 == 0, "16-byte vector reads of the transpose buffer");
static_assert(sizeof(FfShared::xpose) >= 8 * FF_EPW * 16 * 32 * sizeof(float) / 2,
              "the float32 staging of one weight block's epilogue warps fits in the transpose buffer");

// 64-column atoms of the contraction axis a tile of expert e reads: all of K, or (MODE 2
// with per-expert row counts) the atoms that hold the expert's rows, at least one.
template <int MODE>
__device__ __forceinline__ int ff_atoms(const FfnParams& p, int e, int K) {
  if (MODE != 2 || !p.kcount) return K / FF_BK;
  const int n = min(max(p.kcount[e], 0), K);
  return max(1, (n + FF_BK - 1) / FF_BK);
}

template <int MB>
__device__ __forceinline__ void epi_sync() {  // named barrier over the epilogue warps
  asm volatile("bar.sync 1, %0;" ::"n"(128 * FF_EPW * MB) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// MB: 128-row weight blocks per tile, all reading one activation tile (compile-time, so the
// MMA issue loop stays fully unrolled).  NBUF: TMEM accumulator sets (2: the epilogue of
// a tile overlaps the next tile's MMAs; 1 when two sets do not fit in 512 columns).
// MODE 0: the forward (layer 1: + bias, ReLU); both operands K-major.
// MODE 1, the backward's dh = (dye W2) * [h > 0] and dxe = dh W1: the weights are read as
// they are stored (W2 [E, d, F] as layer 1's A with K = d, W1 [E, F, d] as layer 2's with
// K = F), i.e. MN-major A operands; layer 1 keeps the sum where the saved forward activation
// hmask is positive.
// MODE 2, a weight gradient (sum over an expert's rows): both operands MN-major with the
// expert's rows as the contraction axis, read through 4-D tensor maps [E][rows][..] so rows
// past an expert's block read as zero; layer 1 only (p.layer2 = 0), float32 results stored
// straight to out_f32.
// MODE 3, a plain product out[n, m] = sum_k A[k, m] B[n, k]: A MN-major as stored (3-D map,
// like MODE 1's weights), B K-major rows (like the forward's tokens); layer 1 only, float32
// results as in MODE 2.
// PAIR (MODE 0; clusters of 2): a tile is 2 MB 128-row weight blocks (p.MB = 2 MB for the
// ticket order) against one token chunk, MB blocks per CTA.  The even CTA takes the tickets
// and publishes every tile to both CTAs' queues; each CTA loads its weight blocks and half
// of the chunk's token rows; the even CTA issues tcgen05 cta_group::2 MMAs (M = 256: a
// block of each CTA against all N tokens, N / 2 token rows from each CTA's shared memory),
// whose completions arrive on both CTAs' barriers; each CTA's epilogue writes its blocks'
// features, the odd CTA releasing the accumulator and the queue entry on the even CTA's
// barriers.  Per SM the token rows a tile streams are halved.  The library runs MB = 2,
// NBUF = 1 (four blocks per tile); MB = 1, NBUF = 2 measured no faster.
template <int MB, int NBUF, int MODE, bool PAIR = false>
__global__ void __launch_bounds__(ff_threads<MB>(), 1)
    ffn_persistent_kernel(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmX,
                          const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmH,
                          const __grid_constant__ CUtensorMap tmXp, const __grid_constant__ CUtensorMap tmHp,
                          const __grid_constant__ FfnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FfShared& sh = *reinterpret_cast<FfShared*>(ring + FF_RING);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  static_assert(!PAIR || (MODE == 0 && ((MB == 1 && NBUF == 2) || (MB == 2 && NBUF == 1))),
                "CTA pairs: the forward, one or two blocks per CTA");
  const int BN = p.BN, NA = p.NA, STAGES = p.STAGES;
  const int BNC = PAIR ? BN / 2 : BN;  // token rows of a stage in this CTA's shared memory
  const int prk = PAIR ? (int)cluster_ctarank() : 0;
  const bool issuer = prk == 0;  // (pairs) the even CTA takes tickets and issues the MMAs
  const int ACC = MB * BN;  // TMEM columns of one accumulator set
  const int cols = NBUF * ACC;
  const uint32_t TMEM_COLS = cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    for (int i = 0; i < FF_SCHED; ++i) {
      mbar_init(&sh.sfull[i], 1);
      mbar_init(&sh.sempty[i], PAIR ? 3 : 2);  // the MMA issuer and the epilogue (pairs: both epilogues)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.afull[i], 1);
      mbar_init(&sh.aempty[i], PAIR ? 2 : 1);
    }
    sh.abort_flag = 0;
    sh.ep_disc = make_int4(0, 0, 0, 0);
    fence_mbar_init();
    prefetch_tmap(&tmW1);
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW2);
    prefetch_tmap(&tmH);
    prefetch_tmap(&tmXp);
    prefetch_tmap(&tmHp);
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc_pair(&sh.tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&sh.tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (PAIR) cluster_sync();  // both CTAs' barriers are initialised before any remote arrival or copy
  const uint32_t tmem = sh.tmem_slot;
  // layer-1 tiles of an (expert, chunk); pairs count one per CTA and block
  const int MT1 = p.F / (FF_BM * MB);
  griddep_launch_dependents();  // after the TMEM allocation: a dependent grid cannot starve it
  griddep_wait();               // the dispatched rows, row counts and cleared counters

  if (warp == 0 && lane == 0) {
    // ---------------- scheduler + TMA producer
    const uint64_t w_policy = policy_evict_first();  // used when a weight tile is read once
    uint32_t gst = 0;  // stages issued
    int sidx = 0;      // queue entries published (pairs, odd CTA: received)
    while (true) {
      if (sh.abort_flag) break;
      FfTile tl;
      bool has;
      int nv;
      if (issuer) {
        const uint32_t t = atomicAdd(p.next_tile, 1u);
        has = ff_decode(t, p, tl);
        nv = has ? min(BN, p.expert_rows[tl.e] - tl.nc * BN) : 0;
        if (has && nv <= 0) continue;  // empty chunk
        const int qs = sidx % FF_SCHED;
        if (sidx >= FF_SCHED && !mbar_wait(&sh.sempty[qs], ((sidx / FF_SCHED) - 1) & 1)) {
          raise_error(p.err, ERR_TIMEOUT);
          sh.abort_flag = 1;
          break;
        }
        const int4 ent = has ? make_int4(tl.layer, tl.e, tl.mt, tl.nc) : make_int4(-1, 0, 0, 0);
        sh.sched[qs] = ent;
        sh.sched_nv[qs] = nv;
        mbar_arrive(&sh.sfull[qs]);
        if (PAIR) {  // the same entry in the odd CTA's queue, released with the arrival
          const uint32_t q4 = dsmem_addr(&sh.sched[qs], 1u);
          dsmem_st_s32(q4, ent.x);
          dsmem_st_s32(q4 + 4, ent.y);
          dsmem_st_s32(q4 + 8, ent.z);
          dsmem_st_s32(q4 + 12, ent.w);
          dsmem_st_s32(dsmem_addr(&sh.sched_nv[qs], 1u), nv);
          mbar_arrive_remote(&sh.sfull[qs], 1u);
        }
      } else {  // (pairs, odd CTA) the even CTA's entry
        const int qs = sidx % FF_SCHED;
        if (!mbar_wait_cluster(&sh.sfull[qs], (sidx / FF_SCHED) & 1)) {
          raise_error(p.err, ERR_TIMEOUT);
          sh.abort_flag = 1;
          break;
        }
        const int4 ent = sh.sched[qs];
        has = ent.x >= 0;
        tl.layer = ent.x;
        tl.e = ent.y;
        tl.mt = ent.z;
        tl.nc = ent.w;
        nv = sh.sched_nv[qs];
      }
      ++sidx;
      if (!has) break;
      const bool l1 = tl.layer == 0;
      if (!l1) {
        // layer 2 reads h of (e, chunk): wait until every layer-1 tile of it is stored
        const uint32_t* cnt = p.done1 + (size_t)tl.e * p.NCH + tl.nc;
        if (ld_acquire_gpu(cnt) < (uint32_t)MT1) {
          const long long t0 = clock64();
          while (ld_acquire_gpu(cnt) < (uint32_t)MT1) {
            if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
              raise_error(p.err, ERR_TIMEOUT);
              break;
            }
          }
        }
        fence_proxy_async_global();  // order the acquire before the TMA reads of h
      }
      const CUtensorMap* tmA = l1 ? &tmW1 : &tmW2;
      const CUtensorMap* tmB = l1 ? &tmX : &tmH;
      const CUtensorMap* tmBp = l1 ? &tmXp : &tmHp;
      // A chunk filled to at most BN - 64 rows loads its activations as 64-row boxes, only
      // as many as cover its rows (nbox = 0: one box of BN rows)
      const int nt = (nv + 15) & ~15;
      const int nbox = (!PAIR && MODE != 2 && BN > FF_PB && nt <= BN - FF_PB) ? (nt + FF_PB - 1) / FF_PB : 0;
      // (pairs) the even CTA's barrier counts both CTAs' bytes
      const uint32_t tx = nbox ? (uint32_t)(NA * MB * FF_ATOM_A + NA * nbox * FF_PB * FF_BK * 2)
                               : (uint32_t)(PAIR ? 2 * p.stage_bytes : p.stage_bytes);
      const int K = l1 ? p.d : p.F;
      const int M = l1 ? p.F : p.d;
      // (pairs) this CTA's weight block of the tile's two, and its half of the chunk's rows
      const int arow = tl.e * M + (PAIR ? (tl.mt * 2 + prk) * MB : tl.mt * MB) * FF_BM;
      const int brow = tl.e * p.R + tl.nc * BN + (PAIR ? prk * (nt / 2) : 0);
      const int atoms = ff_atoms<MODE>(p, tl.e, K);
      bool ok = true;
      for (int a0 = 0; a0 < atoms; a0 += NA) {
        const int slot = (int)(gst % (uint32_t)STAGES);
        if (gst >= (uint32_t)STAGES && !mbar_wait(&sh.empty[slot], ((gst / STAGES) - 1) & 1)) { ok = false; break; }
        // One 3-D box per operand: NA consecutive 64-column atoms of 128 (or BN) rows, each
        // atom a swizzled [rows x 128 B] block; atoms past K read as zero (never used).
        if (issuer) mbar_arrive_expect_tx(&sh.full[slot], tx);
        uint8_t* stage = ring + (size_t)slot * p.stage_bytes;
        if (PAIR) {  // counted on the even CTA's barrier
          const uint32_t fb = dsmem_addr(&sh.full[slot], 0u);
          tma_load_3d_pair(stage, tmA, fb, 0, arow, a0);
          tma_load_3d_pair(stage + NA * MB * FF_ATOM_A, tmB, fb, 0, brow, a0);
          ++gst;
          continue;
        }
        if (MODE == 2)  // activations, MN-major: K rows a0 .. of expert e, 2 MB chunks of 64 features
          tma_load_4d(stage, tmA, &sh.full[slot], 0, a0 * FF_BK, tl.mt * MB * 2, tl.e);
        else if ((MODE == 1 || MODE == 3) && p.w_evict_first)  // as stored, MN-major: K rows of expert e
          tma_load_3d_hint(stage, tmA, &sh.full[slot], 0, tl.e * K + a0 * FF_BK, tl.mt * MB * 2, w_policy);
        else if (MODE == 1 || MODE == 3)
          tma_load_3d(stage, tmA, &sh.full[slot], 0, tl.e * K + a0 * FF_BK, tl.mt * MB * 2);
        else if (p.w_evict_first)
          tma_load_3d_hint(stage, tmA, &sh.full[slot], 0, arow, a0, w_policy);
        else
          tma_load_3d(stage, tmA, &sh.full[slot], 0, arow, a0);
        uint8_t* sb = stage + NA * MB * FF_ATOM_A;
        if (MODE == 2) {  // expert rows as K, BN / 64 chunks of 64 output rows (past the end: zeros)
          tma_load_4d(sb, tmB, &sh.full[slot], 0, a0 * FF_BK, tl.nc * (BN / 64), tl.e);
        } else if (nbox == 0) {
          tma_load_3d(sb, tmB, &sh.full[slot], 0, brow, a0);
        } else {
          for (int at = 0; at < NA; ++at)  // atom at keeps its [BN x 128 B] place in the stage
            for (int i = 0; i < nbox; ++i)
              tma_load_3d(sb + (size_t)(at * BN + i * FF_PB) * (FF_BK * 2), tmBp, &sh.full[slot], 0,
                          brow + i * FF_PB, a0 + at);
        }
        ++gst;
      }
      if (!ok) {
        raise_error(p.err, ERR_TIMEOUT);
        sh.abort_flag = 1;
        break;
      }
    }
    // Drain: every copy started here has landed before the CTA can leave.  (Pairs: the
    // copies count on the even CTA's barriers; the MMAs' release of each stage, which
    // arrives on this CTA's barriers, follows them, and no arrival is left in flight.  The
    // even CTA also waits for the odd CTA's releases of the last queue entries.)
    for (uint32_t i = gst > (uint32_t)STAGES ? gst - STAGES : 0; i < gst; ++i)
      if (!mbar_wait(PAIR ? &sh.empty[i % STAGES] : &sh.full[i % STAGES], (i / STAGES) & 1))
        raise_error(p.err, ERR_TIMEOUT);
    if (PAIR && issuer && !sh.abort_flag)
      for (int i = sidx > FF_SCHED ? sidx - FF_SCHED : 0; i < sidx - 1; ++i)  // the last entry stops
        if (!mbar_wait(&sh.sempty[i % FF_SCHED], (i / FF_SCHED) & 1)) raise_error(p.err, ERR_TIMEOUT);
  } else if (warp == 1 && lane == 0 && issuer) {
    // ---------------- MMA issuer (pairs: the even CTA, M = 256 over both CTAs' blocks)
    uint32_t gst = 0;
    int sidx = 0, lt = 0;
    while (true) {
      const int qs = sidx % FF_SCHED;
      if (!mbar_wait(&sh.sfull[qs], (sidx / FF_SCHED) & 1)) {
        raise_error(p.err, ERR_TIMEOUT);
        sh.abort_flag = 1;
        break;
      }
      const int4 tv = sh.sched[qs];
      if (tv.x < 0) break;
      // N = the chunk's filled rows rounded up to 16: MMA time and operand reads scale with N.
      // Bits 15 / 16: A / B read MN-major.
      const uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * FF_BM : FF_BM, MODE == 2 ? BN : (sh.sched_nv[qs] + 15) & ~15) |
                             (MODE >= 1 ? (1u << 15) : 0u) | (MODE == 2 ? (1u << 16) : 0u);
      const int buf = lt % NBUF;
      if (lt >= NBUF && !mbar_wait(&sh.aempty[buf], ((lt / NBUF) - 1) & 1)) {
        raise_error(p.err, ERR_TIMEOUT);
        sh.abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int atoms = ff_atoms<MODE>(p, tv.y, tv.x == 0 ? p.d : p.F);
      const uint32_t acc = tmem + (uint32_t)(buf * ACC);
      bool ok = true;
      for (int a0 = 0; a0 < atoms; a0 += NA) {
        const int slot = (int)(gst % (uint32_t)STAGES);
        if (!mbar_wait(&sh.full[slot], (gst / STAGES) & 1)) { ok = false; break; }
        tc_fence_after();
        // Descriptors of the stage's first A and B atoms; later K-steps and atoms add their
        // offset (16-byte units) to the start-address field, which cannot carry out of its
        // 14 bits inside the 227 KB shared window.
        const uint32_t st = smem_u32(ring + (size_t)slot * p.stage_bytes);
        // MN-major boxes hold 64 * NA k-rows per 64-element chunk: chunk stride (LBO) in bytes
        const uint32_t mn_lbo = (uint32_t)(NA * FF_BK * 128);
        const uint64_t da = MODE == 0 ? sw128_kmajor_desc(st) : sw128_mnmajor_desc(st, mn_lbo);
        const uint64_t db = MODE == 2 ? sw128_mnmajor_desc(st + NA * MB * FF_ATOM_A, mn_lbo)
                                      : sw128_kmajor_desc(st + NA * MB * FF_ATOM_A);
        const uint32_t b_atom16 = (uint32_t)(BNC * FF_BK * 2) >> 4;
#pragma unroll
        for (int at = 0; at < 2; ++at) {
          if (at >= NA || a0 + at >= atoms) break;
#pragma unroll
          for (int kk = 0; kk < FF_BK / 16; ++kk)
#pragma unroll
            for (int hb = 0; hb < MB; ++hb) {  // weight block hb: rows 128 hb .. of the atom
              // A: K-major atoms of 128 rows; MN-major: chunks 2 hb, 2 hb + 1, k-row 64 at + 16 kk
              const uint32_t aoff = MODE == 0 ? (uint32_t)((at * MB + hb) * FF_ATOM_A + kk * 32)
                                              : (uint32_t)(2 * hb) * mn_lbo + (uint32_t)((at * FF_BK + kk * 16) * 128);
              const uint32_t boff16 = MODE == 2 ? (uint32_t)(((at * FF_BK + kk * 16) * 128) >> 4)
                                                : at * b_atom16 + (uint32_t)((kk * 32) >> 4);
              if (PAIR)
                tc_mma_bf16_pair(acc + (uint32_t)(hb * BN), da + (uint64_t)(aoff >> 4), db + (uint64_t)boff16,
                                 idesc, (a0 > 0 || at > 0 || kk > 0) ? 1u : 0u);
              else
                tc_mma_bf16(acc + (uint32_t)(hb * BN), da + (uint64_t)(aoff >> 4), db + (uint64_t)boff16, idesc,
                            (a0 > 0 || at > 0 || kk > 0) ? 1u : 0u);
            }
        }
        if (PAIR)
          tc_commit_pair(&sh.empty[slot], (uint16_t)3u);
        else
          tc_commit(&sh.empty[slot]);
        ++gst;
      }
      if (PAIR)
        tc_commit_pair(&sh.afull[buf], (uint16_t)3u);
      else
        tc_commit(&sh.afull[buf]);  // the accumulator is complete once these MMAs are
      if (!ok) {
        raise_error(p.err, ERR_TIMEOUT);
        sh.abort_flag = 1;
        break;
      }
      mbar_arrive(&sh.sempty[qs]);
      ++lt;
      ++sidx;
    }
    // (pairs) both epilogues' releases of the last accumulator sets have arrived before
    // this CTA can leave
    if (PAIR && !sh.abort_flag)
      for (int i = lt > NBUF ? lt - NBUF : 0; i < lt; ++i)
        if (!mbar_wait(&sh.aempty[i % NBUF], (i / NBUF) & 1)) raise_error(p.err, ERR_TIMEOUT);
  } else if (warp >= 2) {
    // ---------------- epilogue (warps 2 .. 1 + 8 MB; TMEM lane quadrant = warp % 4,
    // weight block hb = (warp - 2) / 8, column slice part = ((warp - 2) / 4) % 2)
    const int quad = warp & 3;
    const int hb = (warp - 2) >> 3;
    const int part = ((warp - 2) >> 2) & 1;
    const bool leader = threadIdx.x == 64;
    int sidx = 0, lt = 0;
    while (true) {
      const int qs = sidx % FF_SCHED;
      const int buf = lt % NBUF;
      // The leader takes the tile from the queue and broadcasts it; everyone then starts the
      // tile's bias load (and, for the combine, gathers its tokens and gates) while the
      // leader waits for the accumulator.  Readers of a broadcast are done with it before
      // the end-of-tile barrier, so the leader never overwrites it early.
      if (leader) {
        // (pairs, odd CTA) the entry was stored by the even CTA: a cluster-scope acquire
        const int ok = (PAIR ? mbar_wait_cluster(&sh.sfull[qs], (sidx / FF_SCHED) & 1)
                             : mbar_wait(&sh.sfull[qs], (sidx / FF_SCHED) & 1)) ? 1 : 0;
        if (!ok) {
          raise_error(p.err, ERR_TIMEOUT);
          sh.abort_flag = 1;
        }
        sh.ep_ok = ok;
        sh.ep_tile = sh.sched[qs];
        sh.ep_nv = sh.sched_nv[qs];
      }
      epi_sync<MB>();
      const int4 tv = sh.ep_tile;
      const int nv = sh.ep_nv;
      const int4 dc = sh.ep_disc;  // the leader writes it again only after the next barrier
      if (dc.x) {
        // Nothing reads that chunk's h again: drop its 128-byte lines from L2 without writing
        // them back to DRAM (the rows' contents become undefined).
        const int lines_per_row = p.F * 2 / 128;
        const __nv_bfloat16* h0 = p.h + ((size_t)dc.y * p.R + dc.z) * p.F;
        for (int i = threadIdx.x - 64; i < dc.w * lines_per_row; i += 128 * FF_EPW * MB)
          l2_discard_line(h0 + (size_t)(i / lines_per_row) * p.F + (size_t)(i % lines_per_row) * 64);
      }
      if (!sh.ep_ok || tv.x < 0) break;
      const bool l1 = tv.x == 0;
      const int e = tv.y, mt = tv.z, nc = tv.w;
      const int n0 = nc * BN;
      const int M = l1 ? p.F : p.d;
      const int blk = PAIR ? (mt * 2 + prk) * MB + hb : mt * MB + hb;  // this warp's 128-row weight block
      const int m = blk * FF_BM + quad * 32 + lane;
      const __nv_bfloat16* bias = l1 ? p.b1 : p.b2;
      const float bv = bias ? __bfloat162float(bias[(size_t)e * M + m]) : 0.f;
      const uint32_t taddr = tmem + (uint32_t)(buf * ACC + hb * BN) + ((uint32_t)(quad * 32) << 16);
      if (!l1 && p.combine) {  // the tile's tokens and gates (two dependent loads per column)
        for (int j = threadIdx.x - 64; j < nv; j += 128 * FF_EPW * MB) {
          const int tk = p.tok_of_row[(size_t)e * p.R + n0 + j];
          sh.tok[j] = tk;
          sh.gate[j] = p.gate[tk];
        }
      }
      if (leader) {
        const int ok = mbar_wait(&sh.afull[buf], (lt / NBUF) & 1) ? 1 : 0;
        if (!ok) {
          raise_error(p.err, ERR_TIMEOUT);
          sh.abort_flag = 1;
        }
        sh.ep_acc_ok = ok;
      }
      epi_sync<MB>();  // the accumulator is complete; the combine's tokens and gates are in place
      if (!sh.ep_acc_ok) break;
      tc_fence_after();
      // The two warps of a quadrant take alternate 32-column slices; both TMEM loads of a
      // slice are in flight before one wait.
      if (MODE >= 2) {
        // float32 results, token-major.  Each 16-column chunk goes through shared memory as
        // [16 tokens][32 features] (lane = feature); lane L then stores features 4 (L % 8) ..
        // + 3 of tokens L / 8 + 4 i, i < 4, as 16-byte vectors (8 lanes per 128-byte row).
        float* xf = reinterpret_cast<float*>(&sh.xpose[0][0][0]) + (warp - 2) * (16 * 32);
        const int mb0 = blk * FF_BM + quad * 32;  // first feature of this warp
#pragma unroll 1
        for (int c0 = 32 * part; c0 < nv; c0 += 64) {
          uint32_t r[2][16];
          const int nch = min(2, (nv - c0 + 15) / 16);
#pragma unroll
          for (int q = 0; q < 2; ++q)
            if (q < nch) tmem_ld16(taddr + (uint32_t)(c0 + 16 * q), r[q]);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            if (q >= nch) break;
#pragma unroll
            for (int j = 0; j < 16; ++j) xf[j * 32 + lane] = __uint_as_float(r[q][j]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int j = (lane >> 3) + 4 * i;
              const int col = c0 + 16 * q + j;
              const float4 v = *reinterpret_cast<const float4*>(xf + j * 32 + 4 * (lane & 7));
              if (col < nv)
                *reinterpret_cast<float4*>(p.out_f32 + ((size_t)e * p.R + n0 + col) * p.F + mb0 + 4 * (lane & 7)) = v;
            }
            __syncwarp();  // the chunk's reads of xf are done before the next chunk writes it
          }
        }
      }
#pragma unroll 1
      for (int c0 = 32 * part; MODE < 2 && c0 < nv; c0 += 64) {
        uint32_t r[2][16];
        const int nch = min(2, (nv - c0 + 15) / 16);
#pragma unroll
        for (int q = 0; q < 2; ++q)
          if (q < nch) tmem_ld16(taddr + (uint32_t)(c0 + 16 * q), r[q]);
        tmem_ld_wait();
        // Each 16-column chunk goes through shared memory as 8 token pairs x 32 features, one
        // 32-bit word (both tokens of a pair) per lane and pair; each lane then reads the 8
        // features of one pair and one feature group (two 16-byte loads, the halves swapped on
        // odd pairs so a quarter-warp covers all banks) and splits the two tokens by byte
        // permutes into two 16-byte stores.
        uint32_t* xw = reinterpret_cast<uint32_t*>(&sh.xpose[warp - 2][0][0]);
        const int ip = lane >> 2, f8 = (lane & 3) * 8;
        const int sw = (ip & 1) * 4;
        const int mb = blk * FF_BM + quad * 32;  // first feature of this warp
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (q >= nch) break;
          const int cb = c0 + 16 * q;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float v0 = __uint_as_float(r[q][2 * i]) + bv, v1 = __uint_as_float(r[q][2 * i + 1]) + bv;
            if (l1 && MODE == 0) {
              v0 = fmaxf(v0, 0.f);
              v1 = fmaxf(v1, 0.f);
            }
            const __nv_bfloat162 pr = __floats2bfloat162_rn(v0, v1);  // h, or ye rounded to bf16
            xw[i * 32 + lane] = *reinterpret_cast<const uint32_t*>(&pr);
          }
          __syncwarp();
          const uint4 w0 = *reinterpret_cast<const uint4*>(xw + ip * 32 + f8 + sw);
          const uint4 w1 = *reinterpret_cast<const uint4*>(xw + ip * 32 + f8 + 4 - sw);
          const uint4 lo = sw ? w1 : w0, hi = sw ? w0 : w1;  // features f8 .. +3, f8 + 4 .. +7
          uint4 tv2[2];
          tv2[0] = make_uint4(__byte_perm(lo.x, lo.y, 0x5410), __byte_perm(lo.z, lo.w, 0x5410),
                              __byte_perm(hi.x, hi.y, 0x5410), __byte_perm(hi.z, hi.w, 0x5410));
          tv2[1] = make_uint4(__byte_perm(lo.x, lo.y, 0x7632), __byte_perm(lo.z, lo.w, 0x7632),
                              __byte_perm(hi.x, hi.y, 0x7632), __byte_perm(hi.z, hi.w, 0x7632));
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2) {
            const int j = 2 * ip + t2;
            if (cb + j < nv) {
              uint4 val = tv2[t2];
              const size_t row = (size_t)e * p.R + n0 + cb + j;
              if (MODE == 1 && l1) {
                // dh keeps its value where the saved forward activation h is > 0: the same 8
                // features of h as one 16-byte load, each bf16 kept when its sign is clear and it
                // is not zero
                const uint4 hm = __ldg(reinterpret_cast<const uint4*>(p.hmask + row * p.F + mb + f8));
                const uint32_t hw[4] = {hm.x, hm.y, hm.z, hm.w};
                uint32_t* vw = reinterpret_cast<uint32_t*>(&val);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const uint32_t lo_keep = ((hw[k] & 0x8000u) == 0u && (hw[k] & 0x7fffu) != 0u) ? 0x0000ffffu : 0u;
                  const uint32_t hi_keep = ((hw[k] & 0x80000000u) == 0u && (hw[k] & 0x7fff0000u) != 0u) ? 0xffff0000u : 0u;
                  vw[k] &= lo_keep | hi_keep;
                }
              }
              if (l1) {
                *reinterpret_cast<uint4*>(p.h + row * p.F + mb + f8) = val;
              } else if (!p.combine) {
                *reinterpret_cast<uint4*>(p.out + row * p.d + mb + f8) = val;
              } else {
                // y_t = gate_t * ye (+ x_t): the token and gate of this row, the residual as a vector
                const int tk = sh.tok[cb + j];
                const float g = sh.gate[cb + j];
                const __nv_bfloat162* yv = reinterpret_cast<const __nv_bfloat162*>(&val);
                float o[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float2 f = __bfloat1622float2(yv[k]);
                  o[2 * k] = g * f.x;
                  o[2 * k + 1] = g * f.y;
                }
                if (p.resid) {
                  const uint4 rv = __ldg(reinterpret_cast<const uint4*>(p.resid + (size_t)tk * p.d + mb + f8));
                  const __nv_bfloat162* rr = reinterpret_cast<const __nv_bfloat162*>(&rv);
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    const float2 f = __bfloat1622float2(rr[k]);
                    o[2 * k] += f.x;
                    o[2 * k + 1] += f.y;
                  }
                }
                uint4 ov;
                __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&ov);
#pragma unroll
                for (int k = 0; k < 4; ++k) op[k] = __floats2bfloat162_rn(o[2 * k], o[2 * k + 1]);
                *reinterpret_cast<uint4*>(p.out + (size_t)tk * p.d + mb + f8) = ov;
              }
            }
          }
          __syncwarp();  // the chunk's reads of xw are done before the next chunk writes it
        }
      }
      tc_fence_before();
      epi_sync<MB>();  // every thread's TMEM reads and stores of this tile are done
      if (leader) {
        if (PAIR && !issuer)  // the even CTA's barriers
          mbar_arrive_remote(&sh.aempty[buf], 0u);
        else
          mbar_arrive(&sh.aempty[buf]);
        if (l1 && !(p.stall && e == 0 && mt == 0 && nc == 0)) {
          __threadfence();  // the chunk's h stores (ordered by the barrier) before the count
          atomicAdd(p.done1 + (size_t)e * p.NCH + nc, 1u);
        }
        // Every copy of h this layer-2 tile made had landed before its accumulator was
        // complete; the tile that completes its chunk's count is the chunk's last reader
        // (pairs: the even CTA counts for both).  Off the accumulator's path: counted after
        // the release, the lines dropped while the next tile's MMAs run.
        int last = 0;
        if (!l1 && p.discard_h && issuer) {
          __threadfence();
          last = atomicAdd(p.done2 + (size_t)e * p.NCH + nc, 1u) == (uint32_t)(p.d / (FF_BM * p.MB)) - 1u ? 1 : 0;
          if (last) __threadfence();
        }
        sh.ep_disc = make_int4(last, e, n0, nv);
        if (PAIR && !issuer)
          mbar_arrive_remote(&sh.sempty[qs], 0u);
        else
          mbar_arrive(&sh.sempty[qs]);
      }
      ++lt;
      ++sidx;
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no peer copies into this CTA or arrives on its barriers any more
  if (warp == 1) {
    if (PAIR)
      tmem_dealloc_pair(tmem, TMEM_COLS);
    else
      tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int device_sm_count() {
  static std::atomic<int> cache[64];  // per device; handles on several host threads may fill it
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)FF_BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_3d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_atoms) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || cols % FF_BK != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)FF_BK, rows, cols / FF_BK};
  cuuint64_t strides[2] = {cols * 2, (cuuint64_t)FF_BK * 2};
  cuuint32_t box[3] = {(cuuint32_t)FF_BK, box_rows, box_atoms};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D view [E][rows][cols / 64 chunks][64] of a bf16 buffer [E, rows, cols] (cols % 64 == 0):
// a box {64, box_rows, box_chunks, 1} at (0, r, c, e) holds rows r .. of expert e only (rows
// past `rows` read as zero), chunk by chunk: the MN-major layout with the rows as K.
bool encode_bf16_4d(CUtensorMap* map, const void* base, uint64_t E, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_chunks) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || cols % FF_BK != 0) return false;
  cuuint64_t dims[4] = {(cuuint64_t)FF_BK, rows, cols / FF_BK, E};
  cuuint64_t strides[3] = {cols * 2, (cuuint64_t)FF_BK * 2, rows * cols * 2};
  cuuint32_t box[4] = {(cuuint32_t)FF_BK, box_rows, box_chunks, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_shape_ok(int M, int K) { return M > 0 && K > 0 && M % FF_BM == 0 && K % FF_BK == 0; }

FfnTiling ffn_tiling(int R, int d, int F) {
  FfnTiling t;
  // Chunks of 256 rows (one MMA of N = 256): an expert whose tokens fit one chunk streams
  // its weights once, and a partly filled last chunk loads only the rows it holds.
  t.NCH = R <= 256 ? 1 : (R + 255) / 256;
  t.BN = R > 256 ? 256 : (R <= 16 ? 16 : (R + 15) / 16 * 16);
  // Large token tiles (BN >= 128) are read once for two 128-row weight blocks: TMA ingest
  // per SM (~100 GB/s) is what bounds those layers, and this halves the token re-reads.
  // Small ones keep one block per tile (shorter layer-2 tiles, shorter tail).
  t.MB = (t.BN >= 128 && d % 256 == 0 && F % 256 == 0) ? 2 : 1;
  t.NBUF = 2 * t.MB * t.BN <= 512 ? 2 : 1;
  const int stage_atom = t.MB * FF_ATOM_A + t.BN * FF_BK * 2;
  t.NA = stage_atom <= 48 * 1024 ? 2 : 1;  // 256 contiguous bytes per row when it fits (NA <= 2)
  t.stage_bytes = t.NA * stage_atom;
  t.STAGES = FF_RING / t.stage_bytes < FF_MAX_STAGES ? FF_RING / t.stage_bytes : FF_MAX_STAGES;
  if (t.STAGES < 3 && t.NA == 2) {  // keep at least three stages in flight
    t.NA = 1;
    t.stage_bytes = stage_atom;
    t.STAGES = FF_RING / t.stage_bytes < FF_MAX_STAGES ? FF_RING / t.stage_bytes : FF_MAX_STAGES;
  }
  return t;
}

size_t ffn_counter_words(int E, int R, int d, int F) { return 1 + 2 * (size_t)E * ffn_tiling(R, d, F).NCH; }

// Clusters of 2 of the pair kernel resident at once (cached per device).
static int ffn_pair_clusters(int smem) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(ff_threads<2>(), 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ffn_persistent_kernel<2, 1, 0, true>, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = device_sm_count() / 2;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

int launch_ffn_tc(const FfnLaunch& L, cudaStream_t s, bool pdl) {
  if (L.E == 0 || L.R == 0) return 0;
  if (!tc_shape_ok(L.F, L.d) || (L.mode < 2 && !tc_shape_ok(L.d, L.F))) return -1;
  if (L.mode == 1 && !L.hmask) return -1;
  FfnTiling t = ffn_tiling(L.R, L.d, L.F);
  if (L.mode >= 2 && t.MB == 2) {  // one weight block per tile (one compiled variant each)
    t.MB = 1;
    t.NBUF = 2;
    const int stage_atom = FF_ATOM_A + t.BN * FF_BK * 2;
    t.NA = stage_atom <= 48 * 1024 ? 2 : 1;
    t.stage_bytes = t.NA * stage_atom;
    t.STAGES = FF_RING / t.stage_bytes < FF_MAX_STAGES ? FF_RING / t.stage_bytes : FF_MAX_STAGES;
  }
  if (L.mode == 2 && t.NA == 2) {  // the contraction is one 64-column atom: one atom per box
    t.NA = 1;
    t.stage_bytes = t.MB * FF_ATOM_A + t.BN * FF_BK * 2;
    t.STAGES = FF_RING / t.stage_bytes < FF_MAX_STAGES ? FF_RING / t.stage_bytes : FF_MAX_STAGES;
  }
  // Forward tiles of two weight blocks become tiles of four on CTA pairs: two blocks per
  // CTA, half of the chunk's token rows in each CTA's stages (t.MB = 4 for the ticket order).
  const bool pair = L.mode == 0 && t.MB == 2 && t.BN % 32 == 0 && L.F % 512 == 0 && L.d % 512 == 0;
  if (pair) {
    t.MB = 4;
    t.NBUF = 1;
    const int stage_atom = 2 * FF_ATOM_A + (t.BN / 2) * FF_BK * 2;
    t.NA = stage_atom <= 48 * 1024 ? 2 : 1;
    t.stage_bytes = t.NA * stage_atom;
    t.STAGES = FF_RING / t.stage_bytes < FF_MAX_STAGES ? FF_RING / t.stage_bytes : FF_MAX_STAGES;
    if (t.STAGES < 3 && t.NA == 2) {
      t.NA = 1;
      t.stage_bytes = stage_atom;
      t.STAGES = FF_RING / t.stage_bytes < FF_MAX_STAGES ? FF_RING / t.stage_bytes : FF_MAX_STAGES;
    }
  }
  const int mb_box = pair ? 2 : t.MB;          // weight blocks of a CTA's A boxes
  const int bn_box = pair ? t.BN / 2 : t.BN;   // token rows of a CTA's B boxes
  if (t.STAGES < 2 || t.BN > 256) return -1;
  CUtensorMap tmW1, tmX, tmW2, tmH, tmXp, tmHp;
  if (L.mode == 0) {  // K-major weights [E, M, K]
    if (!encode_bf16_3d(&tmW1, L.W1, (uint64_t)L.E * L.F, (uint64_t)L.d, FF_BM * mb_box, (uint32_t)t.NA)) return -1;
  } else if (L.mode == 1 || L.mode == 3) {  // as stored [E, K, M], MN-major: boxes of 64 NA k-rows x 2 MB chunks
    if (!encode_bf16_3d(&tmW1, L.W1, (uint64_t)L.E * L.d, (uint64_t)L.F, (uint32_t)(FF_BK * t.NA), 2u * t.MB))
      return -1;
  } else {  // activations [E, krows, F] with the rows as K, MN-major
    if (L.krows <= 0 || !encode_bf16_4d(&tmW1, L.W1, (uint64_t)L.E, (uint64_t)L.krows, (uint64_t)L.F, FF_BK, 2u * t.MB))
      return -1;
  }
  if (L.mode == 2) {  // tokens [E, krows, bcols]: the rows as K, BN / 64 chunks of 64 tokens
    const uint64_t bcols = L.bcols > 0 ? (uint64_t)L.bcols : (uint64_t)L.R;
    if (bcols < (uint64_t)L.R || !encode_bf16_4d(&tmX, L.xe, (uint64_t)L.E, (uint64_t)L.krows, bcols, FF_BK,
                                                 (uint32_t)(t.BN / 64)))
      return -1;
  } else if (!encode_bf16_3d(&tmX, L.xe, (uint64_t)L.E * L.R, (uint64_t)L.d, (uint32_t)bn_box, (uint32_t)t.NA)) {
    return -1;
  }
  if (L.mode >= 2) {  // no layer 2: its maps are never read
    tmW2 = tmW1;
    tmH = tmX;
  } else {
    if (L.mode == 1) {
      if (!encode_bf16_3d(&tmW2, L.W2, (uint64_t)L.E * L.F, (uint64_t)L.d, (uint32_t)(FF_BK * t.NA), 2u * t.MB))
        return -1;
    } else if (!encode_bf16_3d(&tmW2, L.W2, (uint64_t)L.E * L.d, (uint64_t)L.F, FF_BM * mb_box, (uint32_t)t.NA)) {
      return -1;
    }
    if (!encode_bf16_3d(&tmH, L.h, (uint64_t)L.E * L.R, (uint64_t)L.F, (uint32_t)bn_box, (uint32_t)t.NA)) return -1;
  }
  if (L.mode != 2 && t.BN > FF_PB) {  // one atom per box: the boxes of a partly filled chunk
    if (!encode_bf16_3d(&tmXp, L.xe, (uint64_t)L.E * L.R, (uint64_t)L.d, (uint32_t)FF_PB, 1u)) return -1;
    if (L.mode == 3)
      tmHp = tmXp;
    else if (!encode_bf16_3d(&tmHp, L.h, (uint64_t)L.E * L.R, (uint64_t)L.F, (uint32_t)FF_PB, 1u))
      return -1;
  } else {
    tmXp = tmX;
    tmHp = tmH;
  }
  FfnParams p{};
  p.b1 = (const __nv_bfloat16*)L.b1;
  p.b2 = (const __nv_bfloat16*)L.b2;
  p.h = (__nv_bfloat16*)L.h;
  p.out = (__nv_bfloat16*)L.out;
  p.expert_rows = L.expert_rows;
  p.tok_of_row = L.tok_of_row;
  p.gate = L.gate;
  p.resid = (const __nv_bfloat16*)L.resid;
  p.next_tile = L.counters;
  p.done1 = L.counters + 1;
  p.done2 = L.counters + 1 + (size_t)L.E * t.NCH;
  p.err = L.err;
  p.E = L.E;
  p.R = L.R;
  p.d = L.d;
  p.F = L.F;
  p.BN = t.BN;
  p.NCH = t.NCH;
  p.MB = t.MB;
  // Layer-2 tiles of an expert are handed out LOOK experts after its layer-1 tiles: a
  // lead of about 8 tiles per CTA, so a layer-1 tile (up to ~3 tiles of queue latency
  // behind a CTA's earlier tiles) is normally stored before anyone needs it.
  const int l2_blocks = L.mode >= 2 ? 0 : L.d / (FF_BM * t.MB);
  const int per_expert = t.NCH * (L.F / (FF_BM * t.MB) + l2_blocks);
  // CTAs of the launch: one per SM (pairs: as many clusters as fit), or the caller's budget
  const int smem = FF_RING + (int)sizeof(FfShared) + 1024;
  int ctas_max = device_sm_count();
  if (pair) {
    // the occupancy query sees the kernel's shared-memory limit, so it is set first
    if (cudaFuncSetAttribute(ffn_persistent_kernel<2, 1, 0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return -1;
    const int fit = 2 * ffn_pair_clusters(smem);
    ctas_max = L.max_ctas > 0 && L.max_ctas < fit ? (L.max_ctas >= 2 ? L.max_ctas / 2 * 2 : 2) : fit;
  } else if (L.max_ctas > 0 && L.max_ctas < ctas_max) {
    ctas_max = L.max_ctas;
  }
  p.LOOK = (8 * ctas_max + per_expert - 1) / per_expert;
  if (p.LOOK > L.E) p.LOOK = L.E;
  if (p.LOOK < 1) p.LOOK = 1;
  p.NA = t.NA;
  p.STAGES = t.STAGES;
  p.stage_bytes = t.stage_bytes;
  p.combine = L.combine ? 1 : 0;
  p.hmask = (const __nv_bfloat16*)L.hmask;
  p.layer2 = L.mode >= 2 ? 0 : 1;
  p.stall = L.stall ? 1 : 0;
  // Dropping h's lines pays where h does not stay in L2 until the next launch overwrites it
  // (its dirty lines would be written back to DRAM: more than half of the 126 MB L2) and the
  // epilogue has slack (two accumulator sets).  Measured: 2048 experts (268 MB of h, two
  // sets) FFN 1942 -> 1905 us, DRAM writes 290 -> 82 MB; with one accumulator set
  // (skewed-e64-g8, switch-large-e128) 228 -> 238 and 533 -> 547 us, so not there.
  const bool big_h = (size_t)L.E * L.R * L.F * 2 > ((size_t)64 << 20);
  p.discard_h = L.mode == 0 && (L.discard_h == 2 || (L.discard_h == 1 && big_h && t.NBUF == 2 && !pair)) ? 1 : 0;
  p.out_f32 = L.out_f32;
  p.kcount = L.mode == 2 ? L.kcount : nullptr;
  if (L.mode >= 2 && !L.out_f32) return -1;
  if (L.mode == 2 && t.BN % 64 != 0) return -1;
  p.w_evict_first = t.NCH == 1 ? 1 : 0;  // several chunks re-read a weight tile
  const long long tiles = (long long)L.E * t.NCH * (L.F / (FF_BM * t.MB) + l2_blocks);
  if (tiles >= (1ll << 31) || (long long)L.E * L.R >= (1ll << 31) || (long long)L.E * L.F >= (1ll << 31) ||
      (long long)L.E * L.d >= (1ll << 31))
    return -1;  // tickets and TMA row coordinates are 32-bit
  cudaError_t e;
  if (pair) {
    auto kern = ffn_persistent_kernel<2, 1, 0, true>;
    const int fit = ctas_max / 2;
    const int pairs = (int)(tiles < fit ? tiles : fit);
    e = launch_k(kern, dim3((unsigned)(2 * pairs)), dim3(ff_threads<2>()), (size_t)smem, s, pdl, 2, tmW1, tmX, tmW2,
                 tmH, tmXp, tmHp, p);
    return e == cudaSuccess ? 1 : -1;
  }
  const int ctas = (int)(tiles < ctas_max ? tiles : ctas_max);
#define SMOE_FFN(MBV, NBV, MK)                                                                                     \
  do {                                                                                                             \
    auto kern = ffn_persistent_kernel<MBV, NBV, MK>;                                                               \
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -1; \
    e = launch_k(kern, dim3((unsigned)ctas), dim3(ff_threads<MBV>()), (size_t)smem, s, pdl, 1, tmW1, tmX, tmW2, tmH, \
                 tmXp, tmHp, p);                                                                                               \
  } while (0)
  if (L.mode == 2) {  // d < 128: one weight block per tile, two accumulator sets
    if (t.MB != 1 || t.NBUF != 2) return -1;
    SMOE_FFN(1, 2, 2);
  } else if (L.mode == 3) {
    if (t.MB != 1 || t.NBUF != 2) return -1;
    SMOE_FFN(1, 2, 3);
  } else if (t.MB == 1) {
    if (L.mode == 1) SMOE_FFN(1, 2, 1); else SMOE_FFN(1, 2, 0);
  } else if (t.NBUF == 2) {
    if (L.mode == 1) SMOE_FFN(2, 2, 1); else SMOE_FFN(2, 2, 0);
  } else {
    if (L.mode == 1) SMOE_FFN(2, 1, 1); else SMOE_FFN(2, 1, 0);
  }
#undef SMOE_FFN
  return e == cudaSuccess ? 1 : -1;
}

}  // namespace smoe
