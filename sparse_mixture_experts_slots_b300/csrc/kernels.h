// Internal launchers of the Switch MoE kernels (host side).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace smoe {

// Launch `kern` on stream s.  pdl: the kernel may start while the previous kernel of the
// stream finishes (it must call griddep_wait() before touching that kernel's results);
// cluster_x > 1: thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                     unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Tokens per routing tile (softmax/top-1 CTA and slot-scan warp).
constexpr int ROUTE_TILE = 128;

struct RouteArgs {
  // inputs
  const void* x;       // [N, d] act
  const float* Wr;     // [E, d]
  const float* br;     // [E] or null
  int G, T, d, E, C, R;
  bool x_bf16;
  float alpha;
  bool debug;
  bool slots;          // false: leave rank in slot[] (a fused dispatch finishes the slots)
  // workspace
  float* logits;       // [N, E] float32 logits of the CUDA-core router (workspace or the caller's)
  float* logits_out;   // [N, E] or null: logits the caller asked for
  void* wsplit;        // W_r split into hi, mid, lo bf16 pieces (tensor-core router; layout in route_tc.cu);
                       // with Wr null the router uses it as it is (prepared by an earlier split)
  void* xchg;          // router_tc_exchange_bytes of zeroed memory (tensor-core router over more than
                       // two expert slices: the slices meet in global memory), or null: clusters
  int32_t* tile_hist;  // [G, nT, E]
  float* tile_P;       // [G, nT, E]
  float* tile_Z;       // [G, nT]: sum over the tile's tokens of (log sum_e exp z)^2
  int32_t* tile_base;  // [G, nT, E]
  int32_t* group_off;  // [G, E]
  int32_t* tok_of_row; // [E * R]
  float* scan_partial; // [G, ceil(E / 32)]
  uint32_t* scan_counter;  // one word, zero between launches
  uint32_t* err;
  // outputs
  int32_t* expert; int32_t* slot; uint8_t* keep; float* gate; int32_t* row;
  int32_t* raw; int32_t* accepted; float* P; float* balance; float* aux_g; float* aux;
  int32_t* expert_rows;
  float* probs;        // or null
  float* z_g;          // [G] router z-loss per group, or null
  float* z;            // [1] its mean over groups, or null
  // top-2 routing (top2): second choices and their per-tile counts / prefixes
  bool top2;
  int32_t* expert2; int32_t* slot2; uint8_t* keep2; float* gate2; int32_t* row2;
  int32_t* raw2; int32_t* accepted2;
  int32_t* tile_hist2; // [G, nT, E]
  int32_t* tile_base2; // [G, nT, E]
  int max_ctas;        // > 0: at most this many CTAs for the persistent tensor-core router (raised
                       // to the fewest its slices need); 0: as many as fit on the device
};

// Batched strided product C_b(i, j) = sum_k A_b(i, k) B_b(j, k) (see backward.cu).
struct BgemmArgs {
  int M, N, K;
  const int32_t* limM; const int32_t* limN; const int32_t* limK;  // per-batch limits or null
  long long Ktot;      // > 0: batch b covers k in [b K, min((b + 1) K, Ktot)) (a split of one K)
  long long sAb, sAi, sAk, sBb, sBj, sBk, sCb, sCi, sCj, sMb, sMi, sMj;
};

// Backward of the top-1 layer (backward.cu); float32 gradients.
struct BackwardArgs {
  int G, T, E, R, d, F;
  bool bf16;           // activations and expert weights bfloat16 (else float32)
  float alpha, w_aux, w_z;
  bool residual;
  // forward inputs and saved activations
  const void* x; const void* dy; const float* Wr; const void* W1; const void* W2;
  const void* xe; const void* h; const void* ye;  // [E, R, d], [E, R, F], [E, R, d]
  const float* logits;                             // [N, E]
  const int32_t* expert; const int32_t* row; const float* gate;
  const int32_t* raw;                              // [G, E] choices before truncation
  const int32_t* expert_rows;                      // [E]
  // outputs (db1, db2, dbr may be null)
  float* dx; float* dWr; float* dbr; float* dW1; float* db1; float* dW2; float* db2;
  // workspace
  float* dye; float* dh; float* dxe; float* dg; float* dz;
  // tensor-core path (bf16, tc_shape_ok): the four expert products on the persistent FFN
  // kernel, reading the weights and the saved activations in place (MN-major operands)
  bool tc;
  void* dye16; void* dh16; void* dxe16;  // [E, R, d], [E, R, F], [E, R, d] bf16
  uint32_t* counters; int counter_words; uint32_t* err;
  // weight gradients on the same kernel (mode 2): expert rows as the contraction axis
  int Rpad;                                   // R rounded up to 64
  int32_t* rows_d; int32_t* rows_F;            // [E] filled with d, F
  uint32_t* counters2; int counter2_words;      // 1 + E * ceil(max(d, F) / 256)
  // split sums over tokens (dWr, dbr): partial products / sums, nsplit of them
  float* part; int nsplit;                      // [nsplit, E, d] floats (>= nsplit * E)
  // router products on the tensor cores (tc, E % 64 == 0): ntc > 0 token chunks of kc rows
  int ntc, kc;
  void* dzp;                                    // [N, 3E] bf16: dz as [hi | lo | hi]
  void* Wp;                                     // [3E, d] bf16: W_r as [hi; hi; lo]
  int32_t* rows_k;                              // [ntc + 1] ints (filled in the backward)
};
int launch_backward(const BackwardArgs& a, cudaStream_t s);

// Blocks of the cross-tile scan (one per 32 experts); scan_partial holds G * this many floats.
__host__ __device__ inline int route_scan_blocks(int E) { return (E + 31) / 32; }

// Router (tensor cores for bf16 x, CUDA cores for float32 x), softmax/top-1, per-tile
// statistics, cross-tile scan + finalize, slots (when a.slots).
// Returns the number of kernels launched (or -1 on a launch error).
int launch_route(const RouteArgs& a, cudaStream_t s);

// Tensor-core router: W_r split + one fused GEMM/softmax/top-1/statistics kernel.
// Writes expert, gate, the in-tile rank (into `rank`), tile_hist, tile_P and, when
// asked, logits_out / probs.  Returns launches or -1.
int launch_router_tc(const RouteArgs& a, int32_t* rank, cudaStream_t s);
// W_r -> its bf16 pieces in wsplit (the first kernel of launch_router_tc when a.Wr is set).
int launch_router_split(const float* Wr, void* wsplit, int E, int d, cudaStream_t s);
int router_tc_experts_per_cta(int E);
// With a.top2 the tensor-core router also takes the second choices (expert2, gate2, the
// in-tile rank of second choices into slot2, tile_hist2) in its own pass: true for up to 1024
// experts (slices of at most 128) and d % 128 == 0.
bool router_tc_top2_fused(int E, int d);
int router_tc_mma_n(int EC);
// Bytes of the split W_r workspace ([Q][d / 64 atoms][hi, mid, lo][EC][64] bf16) for E experts of width d.
size_t router_tc_wsplit_bytes(int E, int d);
// Bytes of the global exchange rows of the tensor-core router for `tiles` 128-token tiles
// (0 when E's slices meet in a cluster).  Zeroed once when allocated.
size_t router_tc_exchange_bytes(long long tiles, int E, bool top2);

// 3-D view [cols / 64 atoms][rows][64] of a row-major bf16 matrix (cols % 64 == 0); a box of
// box_atoms consecutive 64-column atoms of box_rows rows lands as box_atoms swizzled
// [box_rows x 128 B] blocks, one after another.
bool encode_bf16_3d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_atoms);

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// 2-D bf16 tensor map [rows, cols] (cols contiguous), box box_rows x 64 columns, 128-byte swizzle.
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);

// Slots from in-tile ranks, then the dispatch copy (rows staged through shared memory by
// bulk copies).  When y is not null (combine fused into the FFN), dropped tokens' rows of y
// get their final value here (x_residual or zero), and `zero` words at zero_ptr are cleared.
int launch_dispatch_slots(const void* x, void* xe, const RouteArgs& a, void* y, const void* resid,
                          uint32_t* zero_ptr, int zero_words, cudaStream_t s, bool pdl);

// xe[expert[t]*R + row[t]] = x[t] for kept tokens (row[t] >= 0), and likewise for the
// second choice (expert2/row2, top-2 routing; null otherwise); rows r >= expert_rows[e] of
// every expert block are zeroed.
// err: the device error word (a staging wait that runs out sets ERR_TIMEOUT).
int launch_dispatch(const void* x, void* xe, const int32_t* expert, const int32_t* row, const int32_t* expert2,
                    const int32_t* row2, const int32_t* expert_rows, int N, int E, int R, int row_bytes,
                    uint32_t* err, cudaStream_t s);

// y[t] = (row[t] >= 0 ? gate[t] * ye[expert[t]*R + row[t]] : 0)
//        (+ row2[t] >= 0 ? gate2[t] * ye[expert2[t]*R + row2[t]] : 0, top-2) (+ resid[t]).
int launch_combine(const void* ye, const int32_t* expert, const int32_t* row, const float* gate,
                   const int32_t* expert2, const int32_t* row2, const float* gate2, const void* resid,
                   void* y, int N, int d, int E, int R, bool bf16, uint32_t* err, cudaStream_t s, bool pdl);

// out[e*R + n, m] = act(sum_k in[e*R + n, k] * W[e, m, k] + bias[e, m]) for n < expert_rows[e].
// CUDA-core kernel for float32 and for shapes the tensor-core kernel does not take.
int launch_grouped_linear_simt(const void* in, const void* W, const void* bias, void* out,
                               const int32_t* expert_rows, int E, int R, int M, int K, bool relu,
                               bool bf16, cudaStream_t s, bool pdl);

// Expert FFN (both layers of every expert) in one persistent tensor-core kernel.
struct FfnTiling {
  int BN;           // token rows per tile (MMA N), multiple of 16
  int MB;           // 128-row weight blocks per tile (1 or 2)
  int NBUF;         // TMEM accumulator sets (2: double-buffered)
  int NCH;          // chunks of BN rows per expert block
  int NA;           // 64-column atoms per pipeline stage
  int stage_bytes;
  int STAGES;
};
FfnTiling ffn_tiling(int R, int d, int F);
// 32-bit words of scheduler state the kernel needs zeroed at launch.
size_t ffn_counter_words(int E, int R, int d, int F);

struct FfnLaunch {
  const void* xe;            // [E * R, d] bf16
  const void* W1; const void* b1;  // [E, F, d], [E, F] or null
  const void* W2; const void* b2;  // [E, d, F], [E, d] or null
  void* h;                   // [E * R, F] bf16 scratch
  void* out;                 // ye [E * R, d], or y [N, d] when combine
  const int32_t* expert_rows;
  bool combine;
  const int32_t* tok_of_row; // [E * R] (combine)
  const float* gate;         // [N] (combine)
  const void* resid;         // [N, d] or null (combine)
  const void* hmask;         // [E * R, F] (mode 1): layer 1 keeps its sum where hmask > 0
  int mode;                  // 0 forward; 1 backward dh -> dxe (W1 = W2 [E, d, F] and W2 = W1 [E, F, d]
                             // as stored, mask, no bias/ReLU); 2 weight gradient (layer 1 only,
                             // plain sum: W1 = activations [E, krows, F], xe = [E, krows, R],
                             // d = krows rounded up to 64, float32 result in out_f32 [E * R, F])
  int krows;                 // mode 2: rows per expert of W1 / xe (the contraction axis)
  int bcols;                 // mode 2: row length of xe in elements when it is wider than R (else 0)
  float* out_f32;            // modes 2 and 3 output
  const int32_t* kcount;     // mode 2 (or null): rows of each expert on the contraction axis; only the
                             // 64-row atoms holding them are read (rows past the count in the last
                             // one must be zero; an expert with none reads one atom of zeros)
                             // mode 3: out_f32[E * R, F] = sum_k W1[e, k, f] xe[e * R + n, k] (W1 as
                             // stored [E, d, F], xe K-major rows [E * R, d]; layer 1 only)
  uint32_t* counters;        // ffn_counter_words(E, R) words, zero at launch
  uint32_t* err;
  int E, R, d, F;
  bool stall;                // test only: layer-1 tile (expert 0, chunk 0, block 0) never publishes
  int max_ctas;              // > 0: at most this many CTAs (at least one, or one pair); 0: one per SM
  int discard_h;             // mode 0, h not read after this launch (no training): 1 drop its lines
                             // from L2 once the last layer-2 tile of a chunk read them, where h
                             // outgrows half of L2 and the tiles keep two accumulator sets;
                             // 2 for every shape (tests)
};
// Needs d % 128 == 0 and F % 128 == 0 (tc_shape_ok both ways).  Returns launches or -1.
bool tc_shape_ok(int M, int K);
int launch_ffn_tc(const FfnLaunch& L, cudaStream_t s, bool pdl);

// Expert parallelism (ep.cu): chunk[W][El][R] rows <-> packed[El][W R] rows, per-(source,
// expert) counts [W][El]; forward also writes the packed row count per expert (rows_out).
int launch_ep_regroup(const void* src, void* dst, const int32_t* counts, int32_t* rows_out, int W, int El, int R,
                      int row_bytes, bool inverse, cudaStream_t s);

}  // namespace smoe
