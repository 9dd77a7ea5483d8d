// Backward of the top-1 layer: gradients of L = sum(dy * y) + w_aux * aux + w_z * z_loss
// with the choices, slots and capacity mask of the forward held fixed.
//
//   combine:  dye[e, r] = g_t * dy_t for the kept token t in row r of expert e, and
//             dg_t = <dy_t, ye[e, r]> (the gate's gradient; 0 for dropped tokens)
//   experts:  dh = (dye W2_e) * [h > 0];  dW2_e = dye^T h;  db2_e = sum_r dye
//             dxe = dh W1_e;  dW1_e = dh^T xe;  db1_e = sum_r dh
//   router:   dp_te = [e = e*_t] dg_t + w_aux alpha E f_ge / (G T)   (through P, not f)
//             dz_t = p_t * (dp_t - <p_t, dp_t>) + w_z 2 lse_t / (G T) * p_t
//             dWr = dz^T x;  dbr = sum_t dz_t;  dx = dz Wr + dxe[e*_t, row_t] (+ dy)
// The gate keeps the router differentiable (Switch Transformers card, section 方法适配);
// the aux loss's gradient flows through P and not through the hard counts f, and the z-loss
// through the log-sum-exp (070 page, section 核心思想与公式).
//
// With bfloat16 and tensor-core shapes the four expert products run on the persistent
// tcgen05 FFN kernel (ffn_tc.cu) with no copy of any operand: dh -> dxe as its two layers
// reading W2 and W1 as stored (MN-major operands; mode 1, a mask epilogue), dW2 and dW1 as
// layer-1-only launches whose contraction axis is an expert's rows, read MN-major from the
// saved activations (mode 2), with float32 results stored directly.  The rows past each
// expert's count are zeroed first, so they add nothing to those sums.  The router's
// products, and every product for float32 or other widths, run in one batched float32
// kernel on CUDA cores with arbitrary strides and per-batch limits on M, N or K.
#include "common.cuh"
#include "kernels.h"

namespace smoe {

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- batched strided GEMM
// C_b(i, j) = sum_k A_b(i, k) B_b(j, k) for i < M_b, j < N_b, k < K_b, where X_b(u, v) =
// X[b sXb + u sXu + v sXv] and M_b = min(M, limM[b]) (likewise N, K) when a limit array is
// given.  EPI 1: C *= (mask_b(i, j) > 0), the mask in float32 or bfloat16.  ACC: C += .
constexpr int BG_N = 128, BG_K = 16, BG_THREADS = 256;

// Loads one BK-deep slice of an operand tile (rows u < ROWS of the tile, k < BG_K) into
// registers: consecutive threads walk the operand's contiguous axis (k when its k stride
// is 1, else the row axis), so a warp reads whole runs of memory.
template <typename T, int ROWS>
__device__ __forceinline__ void bg_load(const T* __restrict__ X, long long su, long long sk, int u0, int k0, int lim_u,
                                        int lim_k, bool kfast, float (&r)[ROWS * BG_K / BG_THREADS]) {
#pragma unroll
  for (int q = 0; q < ROWS * BG_K / BG_THREADS; ++q) {
    const int idx = threadIdx.x + BG_THREADS * q;
    const int kk = kfast ? idx % BG_K : idx / ROWS;
    const int u = kfast ? idx / BG_K : idx % ROWS;
    const int gu = u0 + u, gk = k0 + kk;
    r[q] = (gu < lim_u && gk < lim_k) ? to_f<T>(X[(long long)gu * su + (long long)gk * sk]) : 0.f;
  }
}
template <int ROWS>
__device__ __forceinline__ void bg_store(float (*S)[ROWS + 4], bool kfast, const float (&r)[ROWS * BG_K / BG_THREADS]) {
#pragma unroll
  for (int q = 0; q < ROWS * BG_K / BG_THREADS; ++q) {
    const int idx = threadIdx.x + BG_THREADS * q;
    const int kk = kfast ? idx % BG_K : idx / ROWS;
    const int u = kfast ? idx / BG_K : idx % ROWS;
    S[kk][u] = r[q];
  }
}

// Tile BM x 128 (BM = 64 or 128), 256 threads in a 16 x 16 grid, each BM/16 rows x 8 columns
// (rows ty + 16 p, columns tx + 16 q); the next K slice is loaded into registers while the
// current one is multiplied.
template <typename TA, typename TB, typename TM, int EPI, bool ACC, int BM>
__global__ void __launch_bounds__(BG_THREADS) bgemm_kernel(const TA* __restrict__ A, const TB* __restrict__ B,
                                                           float* __restrict__ C, const TM* __restrict__ mask,
                                                           BgemmArgs g) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int RA = BM * BG_K / BG_THREADS, RB = BG_N * BG_K / BG_THREADS, PM = BM / 16;
  __shared__ float As[BG_K][BM + 4], Bs[BG_K][BG_N + 4];
  const int b = blockIdx.z;
  const int Mb = g.limM ? min(g.M, g.limM[b]) : g.M;
  const int Nb = g.limN ? min(g.N, g.limN[b]) : g.N;
  int Kb = g.limK ? min(g.K, g.limK[b]) : g.K;
  if (g.Ktot > 0) Kb = (int)min((long long)Kb, g.Ktot - (long long)b * g.K);
  const int i0 = blockIdx.y * BM, j0 = blockIdx.x * BG_N;
  if (i0 >= Mb || j0 >= Nb) return;
  const TA* Ab = A + (long long)b * g.sAb;
  const TB* Bb = B + (long long)b * g.sBb;
  const bool akf = g.sAk == 1, bkf = g.sBk == 1;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[PM][8] = {};
  float ra[RA], rb[RB];
  bg_load<TA, BM>(Ab, g.sAi, g.sAk, i0, 0, Mb, Kb, akf, ra);
  bg_load<TB, BG_N>(Bb, g.sBj, g.sBk, j0, 0, Nb, Kb, bkf, rb);
  for (int k0 = 0; k0 < Kb; k0 += BG_K) {
    bg_store<BM>(As, akf, ra);
    bg_store<BG_N>(Bs, bkf, rb);
    __syncthreads();
    if (k0 + BG_K < Kb) {  // next slice in flight during the products below
      bg_load<TA, BM>(Ab, g.sAi, g.sAk, i0, k0 + BG_K, Mb, Kb, akf, ra);
      bg_load<TB, BG_N>(Bb, g.sBj, g.sBk, j0, k0 + BG_K, Nb, Kb, bkf, rb);
    }
#pragma unroll
    for (int kk = 0; kk < BG_K; ++kk) {
      float a[PM], bv[8];
#pragma unroll
      for (int p = 0; p < PM; ++p) a[p] = As[kk][ty + 16 * p];
#pragma unroll
      for (int q = 0; q < 8; ++q) bv[q] = Bs[kk][tx + 16 * q];
#pragma unroll
      for (int p = 0; p < PM; ++p)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[p][q] = fmaf(a[p], bv[q], acc[p][q]);
    }
    __syncthreads();
  }
  float* Cb = C + (long long)b * g.sCb;
#pragma unroll
  for (int p = 0; p < PM; ++p) {
    const int i = i0 + ty + 16 * p;
    if (i >= Mb) continue;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = j0 + tx + 16 * q;
      if (j >= Nb) continue;
      float v = acc[p][q];
      if (EPI == 1) {
        const TM mv = mask[(long long)b * g.sMb + (long long)i * g.sMi + (long long)j * g.sMj];
        v = to_f<TM>(mv) > 0.f ? v : 0.f;
      }
      float* dst = Cb + (long long)i * g.sCi + (long long)j * g.sCj;
      *dst = ACC ? *dst + v : v;
    }
  }
}

template <typename TA, typename TB, typename TM, int EPI, bool ACC>
static int launch_bg(const TA* A, const TB* B, float* C, const TM* mask, const BgemmArgs& g, int batches,
                     cudaStream_t s) {
  if (g.M <= 0 || g.N <= 0 || batches <= 0) return 0;
  const bool big = g.M >= 128;
  const int BM = big ? 128 : 64;
  const dim3 grid((unsigned)((g.N + BG_N - 1) / BG_N), (unsigned)((g.M + BM - 1) / BM), (unsigned)batches);
  const cudaError_t e =
      big ? launch_k(bgemm_kernel<TA, TB, TM, EPI, ACC, 128>, grid, dim3(BG_THREADS), 0, s, false, 1, A, B, C, mask, g)
          : launch_k(bgemm_kernel<TA, TB, TM, EPI, ACC, 64>, grid, dim3(BG_THREADS), 0, s, false, 1, A, B, C, mask, g);
  return e == cudaSuccess ? 1 : -1;
}

// ---------------------------------------------------------------- combine backward
// Warp per token: dye row = g dy (float32), dg = <dy, ye row>.
template <typename T>
__global__ void __launch_bounds__(256) combine_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ ye,
                                                          const int32_t* __restrict__ expert,
                                                          const int32_t* __restrict__ row,
                                                          const float* __restrict__ gate, float* __restrict__ dye,
                                                          __nv_bfloat16* __restrict__ dye16,
                                                          float* __restrict__ dg, long long N, int d, int R) {
  griddep_wait();
  griddep_launch_dependents();
  const long long t = (long long)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (t >= N) return;
  const int r = row[t];
  if (r < 0) {
    if (lane == 0) dg[t] = 0.f;
    return;
  }
  const long long base = ((long long)expert[t] * R + r) * d;
  const float g = gate[t];
  float s = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float v = to_f<T>(dy[t * d + c]);
    dye[base + c] = g * v;
    if (dye16) dye16[base + c] = __float2bfloat16_rn(g * v);
    s = fmaf(v, to_f<T>(ye[base + c]), s);
  }
  s = warp_sum(s);
  if (lane == 0) dg[t] = s;
}

// ---------------------------------------------------------------- column sums over an expert's rows
// out[e, c] = sum_{r < rows[e]} in[e, r, c] (fixed order), thread per (e, c).
template <typename TI>
__global__ void __launch_bounds__(256) colsum_rows_kernel(const TI* __restrict__ in, const int32_t* __restrict__ rows,
                                                          float* __restrict__ out, int E, int R, int W) {
  griddep_wait();
  griddep_launch_dependents();
  const long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= (long long)E * W) return;
  const int e = (int)(k / W), c = (int)(k % W);
  const int n = rows ? min(R, rows[e]) : R;
  float s = 0.f;
  for (int r = 0; r < n; ++r) s += to_f<TI>(in[((long long)e * R + r) * W + c]);
  out[k] = s;
}

// The same sums with 8 row groups per block and 16-byte column vectors: thread (g, v) of a
// block adds rows g, g + 8, ... of V consecutive columns; the 8 groups' partials are then
// added in group order (fixed order).  Needs W % V == 0 and 16-byte aligned rows.
template <typename TI>
__global__ void __launch_bounds__(256) colsum_rows_vec_kernel(const TI* __restrict__ in, const int32_t* __restrict__ rows,
                                                              float* __restrict__ out, int E, int R, int W) {
  constexpr int V = 16 / sizeof(TI);
  __shared__ float part[8][32 * V];
  griddep_wait();
  griddep_launch_dependents();
  const int e = blockIdx.y;
  const int v = threadIdx.x & 31, g = threadIdx.x >> 5;
  const long long c0 = ((long long)blockIdx.x * 32 + v) * V;
  const int n = rows ? min(R, rows[e]) : R;
  float acc[V];
#pragma unroll
  for (int j = 0; j < V; ++j) acc[j] = 0.f;
  if (c0 < W) {
    const TI* src = in + (long long)e * R * W + c0;
#pragma unroll 4
    for (int r = g; r < n; r += 8) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(src + (long long)r * W));
      const TI* t = reinterpret_cast<const TI*>(&q);
#pragma unroll
      for (int j = 0; j < V; ++j) acc[j] += to_f<TI>(t[j]);
    }
  }
#pragma unroll
  for (int j = 0; j < V; ++j) part[g][v * V + j] = acc[j];
  __syncthreads();
  for (int k = threadIdx.x; k < 32 * V; k += blockDim.x) {
    const long long c = (long long)blockIdx.x * 32 * V + k;
    if (c >= W) continue;
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) t += part[q][k];
    out[(long long)e * W + c] = t;
  }
}

// out[e, c] = sum_{r < rows[e]} in[e, r, c]: the vector kernel when the rows allow it.
template <typename TI>
static cudaError_t launch_colsum_rows(const TI* in, const int32_t* rows, float* out, int E, int R, int W,
                                      cudaStream_t s) {
  constexpr int V = 16 / sizeof(TI);
  if (W % V == 0 && (reinterpret_cast<uintptr_t>(in) & 15u) == 0) {
    const long long bx = ((long long)W + 32 * V - 1) / (32 * V);
    return launch_k(colsum_rows_vec_kernel<TI>, dim3((unsigned)bx, (unsigned)E), dim3(256), 0, s, false, 1, in, rows,
                    out, E, R, W);
  }
  return launch_k(colsum_rows_kernel<TI>, dim3((unsigned)(((long long)E * W + 255) / 256)), dim3(256), 0, s, false, 1,
                  in, rows, out, E, R, W);
}

// ---------------------------------------------------------------- router backward
// Warp per token: p from the logits, dp = onehot(e*) dg + w_aux alpha E f / (G T), the
// softmax Jacobian, plus the z-loss term; writes dz [N, E].
// dzp (or null): dz also as bfloat16 pieces [N, 3E] = [hi | lo | hi] (hi = bf16(dz), lo =
// bf16(dz - hi)) for the tensor-core products dWr and dx.
__global__ void __launch_bounds__(256) router_bwd_kernel(const float* __restrict__ z, const int32_t* __restrict__ expert,
                                                         const float* __restrict__ dg, const int32_t* __restrict__ raw,
                                                         float* __restrict__ dz, __nv_bfloat16* __restrict__ dzp,
                                                         long long N, int T, int E, int G, float aux_coef, float z_coef) {
  griddep_wait();
  griddep_launch_dependents();
  const long long t = (long long)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (t >= N) return;
  const float* zr = z + t * E;
  const int g = (int)(t / T);
  float m = -INFINITY;
  for (int e = lane; e < E; e += 32) m = fmaxf(m, zr[e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  for (int e = lane; e < E; e += 32) s += expf(zr[e] - m);
  s = warp_sum(s);
  const float lse = m + logf(s);
  const int a = expert[t];
  const float dgt = dg[t];
  const int32_t* rg = raw + (long long)g * E;
  // <p, dp>
  float pdp = 0.f;
  for (int e = lane; e < E; e += 32) {
    const float p = expf(zr[e] - m) / s;
    const float dp = (e == a ? dgt : 0.f) + aux_coef * (float)rg[e];
    pdp = fmaf(p, dp, pdp);
  }
  pdp = warp_sum(pdp);
  for (int e = lane; e < E; e += 32) {
    const float p = expf(zr[e] - m) / s;
    const float dp = (e == a ? dgt : 0.f) + aux_coef * (float)rg[e];
    const float v = p * (dp - pdp) + z_coef * lse * p;
    dz[t * E + e] = v;
    if (dzp) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
      __nv_bfloat16* row = dzp + t * 3 * E;
      row[e] = hi;
      row[E + e] = lo;
      row[2 * E + e] = hi;
    }
  }
}

// W_r [E, d] float32 -> Wp [3E, d] bfloat16 = [hi; hi; lo]: with dzp's [hi | lo | hi] the
// product over 3E sums dz_hi W_hi + dz_lo W_hi + dz_hi W_lo (dx = dz W_r to ~2^-16).
__global__ void __launch_bounds__(256) split_wr3_kernel(const float* __restrict__ Wr, __nv_bfloat16* __restrict__ Wp,
                                                        long long n /* E * d */) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const float w = Wr[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    Wp[i] = hi;
    Wp[n + i] = hi;
    Wp[2 * n + i] = __float2bfloat16_rn(w - __bfloat162float(hi));
  }
}

// ---------------------------------------------------------------- dx assembly
// dx_t += dxe[e*_t, row_t] (kept tokens) (+ dy_t with the residual)
template <typename T, typename TX>
__global__ void __launch_bounds__(256) dx_assemble_kernel(float* __restrict__ dx, const TX* __restrict__ dxe,
                                                          const T* __restrict__ dy, const int32_t* __restrict__ expert,
                                                          const int32_t* __restrict__ row, long long N, int d, int R,
                                                          int residual) {
  griddep_wait();
  griddep_launch_dependents();
  const long long t = (long long)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (t >= N) return;
  const int r = row[t];
  const TX* src = r >= 0 ? dxe + ((long long)expert[t] * R + r) * d : nullptr;
  for (int c = lane; c < d; c += 32) {
    float v = dx[t * d + c];
    if (src) v += to_f<TX>(src[c]);
    if (residual) v += to_f<T>(dy[t * d + c]);
    dx[t * d + c] = v;
  }
}

// part[s][c] = sum of in[t][c] over the tokens t of chunk s (kc tokens each, the last one
// shorter): thread per (chunk, column).
__global__ void __launch_bounds__(256) colsum_split_kernel(const float* __restrict__ in, float* __restrict__ part,
                                                           long long N, int W, int kc) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int sidx = blockIdx.y;
  if (c >= W) return;
  const long long t0 = (long long)sidx * kc;
  const long long t1 = min(N, t0 + kc);
  float acc = 0.f;
  for (long long t = t0; t < t1; ++t) acc += in[t * W + c];
  part[(long long)sidx * W + c] = acc;
}

// Rows from rows[e] to the end of its last 64-row atom (rows 0 .. 63 when rows[e] = 0) of
// every expert block of up to three bfloat16 buffers [E, R, w_k] are set to zero: the
// weight-gradient products read whole atoms up to there.  Warp per (expert, row), 16-byte
// stores (w_k % 8 == 0).
__global__ void __launch_bounds__(256) zero_tail_rows_kernel(const int32_t* __restrict__ rows, int E, int R,
                                                             __nv_bfloat16* a, int wa, __nv_bfloat16* b, int wb,
                                                             __nv_bfloat16* c, int wc) {
  const long long w = (long long)blockIdx.x * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (w >= (long long)E * R) return;
  const int e = (int)(w / R), r = (int)(w % R);
  const int n = rows[e];
  if (r < n || r >= 64 * max(1, (n + 63) / 64)) return;  // only the rest of the last 64-row atom
  const uint4 zero = make_uint4(0, 0, 0, 0);
  __nv_bfloat16* bufs[3] = {a, b, c};
  const int widths[3] = {wa, wb, wc};
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    if (!bufs[k]) continue;
    uint4* row = reinterpret_cast<uint4*>(bufs[k] + (size_t)w * widths[k]);
    for (int v = lane; v < widths[k] / 8; v += 32) row[v] = zero;
  }
}

__global__ void fill_i32_kernel(int32_t* __restrict__ a, int n, int v) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) a[i] = v;
}

// ---------------------------------------------------------------- launcher
template <typename T>
static int run_backward(const BackwardArgs& a, cudaStream_t s) {
  const long long N = (long long)a.G * a.T;
  const int E = a.E, R = a.R, d = a.d, F = a.F;
  int n = 0, k;
  const T* x = static_cast<const T*>(a.x);
  const T* dy = static_cast<const T*>(a.dy);
  const T* W1 = static_cast<const T*>(a.W1);
  const T* W2 = static_cast<const T*>(a.W2);
  const T* xe = static_cast<const T*>(a.xe);
  const T* hb = static_cast<const T*>(a.h);
  const T* ye = static_cast<const T*>(a.ye);
#define BW_STEP(expr) \
  do {                \
    k = (expr);       \
    if (k < 0) return -1; \
    n += k;           \
  } while (0)
  if (N > 0)
    BW_STEP(launch_k(combine_bwd_kernel<T>, dim3((unsigned)((N + 7) / 8)), dim3(256), 0, s, false, 1, dy, ye,
                     a.expert, a.row, a.gate, a.dye, (__nv_bfloat16*)a.dye16, a.dg, N, d, R) == cudaSuccess ? 1 : -1);
  const bool tc = a.tc;
  if (tc) {
    // rows past each expert's count hold stale values in h, dye and dh: zero them, so the
    // weight gradients (sums over an expert's rows) read zeros there
    if ((long long)E * R > 0) {
      zero_tail_rows_kernel<<<(unsigned)(((long long)E * R + 7) / 8), 256, 0, s>>>(
          a.expert_rows, E, R, (__nv_bfloat16*)const_cast<void*>(a.h), F, (__nv_bfloat16*)a.dye16, d,
          (__nv_bfloat16*)a.dh16, F);
      if (cudaGetLastError() != cudaSuccess) return -1;
      ++n;
    }
    // dh = (dye W2_e) * [h > 0] and dxe = dh W1_e: the forward's two layers with W2 [E, d, F]
    // and W1 [E, F, d] read as they are stored (MN-major A operands)
    if (cudaMemsetAsync(a.counters, 0, (size_t)a.counter_words * sizeof(uint32_t), s) != cudaSuccess) return -1;
    FfnLaunch L{};
    L.xe = a.dye16;
    L.W1 = a.W2;
    L.W2 = a.W1;
    L.h = a.dh16;
    L.out = a.dxe16;
    L.expert_rows = a.expert_rows;
    L.combine = false;
    L.hmask = a.h;
    L.mode = 1;
    L.counters = a.counters;
    L.err = a.err;
    L.E = E;
    L.R = R;
    L.d = d;
    L.F = F;
    if (R > 0) {
      BW_STEP(launch_ffn_tc(L, s, false));
      // dW2_e = dye^T h and dW1_e = dh^T xe: the contraction axis is an expert's rows, read
      // MN-major from [E, R, .] (only the atoms holding the expert's rows; the rest of the
      // last one zeroed above);
      // float32 results straight into dW2 [E, d, F] and dW1 [E, F, d]
      fill_i32_kernel<<<(E + 255) / 256, 256, 0, s>>>(a.rows_d, E, d);
      fill_i32_kernel<<<(E + 255) / 256, 256, 0, s>>>(a.rows_F, E, F);
      if (cudaGetLastError() != cudaSuccess) return -1;
      n += 2;
      for (int wgt = 0; wgt < 2; ++wgt) {
        // wgt 0: dW2[e, c, f] = sum_r h[r, f] dye[r, c]  (tokens c < d, features f < F)
        // wgt 1: dW1[e, f, c] = sum_r xe[r, c] dh[r, f]  (tokens f < F, features c < d)
        if (cudaMemsetAsync(a.counters2, 0, (size_t)a.counter2_words * sizeof(uint32_t), s) != cudaSuccess) return -1;
        FfnLaunch M{};
        M.W1 = wgt == 0 ? a.h : a.xe;        // A: features
        M.W2 = M.W1;
        M.xe = wgt == 0 ? (const void*)a.dye16 : (const void*)a.dh16;  // B: tokens
        M.expert_rows = wgt == 0 ? a.rows_d : a.rows_F;
        M.kcount = a.expert_rows;            // contraction: only the atoms holding the expert's rows
        M.combine = false;
        M.mode = 2;
        M.counters = a.counters2;
        M.err = a.err;
        M.E = E;
        M.R = wgt == 0 ? d : F;              // tokens per expert
        M.F = wgt == 0 ? F : d;              // features
        M.d = a.Rpad;                        // contraction: the expert's rows, rounded up to 64
        M.krows = R;
        M.out_f32 = wgt == 0 ? a.dW2 : a.dW1;
        BW_STEP(launch_ffn_tc(M, s, false));
      }
    } else {  // no expert rows: the weight gradients are zero
      if (cudaMemsetAsync(a.dW1, 0, (size_t)E * F * d * sizeof(float), s) != cudaSuccess ||
          cudaMemsetAsync(a.dW2, 0, (size_t)E * F * d * sizeof(float), s) != cudaSuccess)
        return -1;
    }
  }
  // dh = (dye W2_e) * [h > 0]: i = row (<= rows_e), j = f, k = c
  if (!tc) {
    BgemmArgs g{};
    g.M = R; g.N = F; g.K = d; g.limM = a.expert_rows;
    g.sAb = (long long)R * d; g.sAi = d; g.sAk = 1;                // dye [E, R, d]
    g.sBb = (long long)d * F; g.sBj = 1; g.sBk = F;                // W2 [E, d, F]: B(j = f, k = c) = W2[c, f]
    g.sCb = (long long)R * F; g.sCi = F; g.sCj = 1;                // dh [E, R, F]
    g.sMb = (long long)R * F; g.sMi = F; g.sMj = 1;                // h
    BW_STEP((launch_bg<float, T, T, 1, false>(a.dye, W2, a.dh, hb, g, E, s)));
  }
  // dW2_e = dye^T h: i = c (d), j = f, k = row (< rows_e)
  {
    BgemmArgs g{};
    g.M = d; g.N = F; g.K = R; g.limK = a.expert_rows;
    g.sAb = (long long)R * d; g.sAi = 1; g.sAk = d;
    g.sBb = (long long)R * F; g.sBj = 1; g.sBk = F;
    g.sCb = (long long)d * F; g.sCi = F; g.sCj = 1;
    if (!tc) BW_STEP((launch_bg<float, T, float, 0, false>(a.dye, hb, a.dW2, nullptr, g, E, s)));
  }
  // dxe = dh W1_e: i = row, j = c, k = f
  if (!tc) {
    BgemmArgs g{};
    g.M = R; g.N = d; g.K = F; g.limM = a.expert_rows;
    g.sAb = (long long)R * F; g.sAi = F; g.sAk = 1;
    g.sBb = (long long)F * d; g.sBj = 1; g.sBk = d;                // W1 [E, F, d]: B(j = c, k = f) = W1[f, c]
    g.sCb = (long long)R * d; g.sCi = d; g.sCj = 1;
    BW_STEP((launch_bg<float, T, float, 0, false>(a.dh, W1, a.dxe, nullptr, g, E, s)));
  }
  // dW1_e = dh^T xe: i = f, j = c, k = row
  {
    BgemmArgs g{};
    g.M = F; g.N = d; g.K = R; g.limK = a.expert_rows;
    g.sAb = (long long)R * F; g.sAi = 1; g.sAk = F;
    g.sBb = (long long)R * d; g.sBj = 1; g.sBk = d;
    g.sCb = (long long)F * d; g.sCi = d; g.sCj = 1;
    if (!tc) BW_STEP((launch_bg<float, T, float, 0, false>(a.dh, xe, a.dW1, nullptr, g, E, s)));
  }
  // bias gradients
  if (a.db2)
    BW_STEP(launch_colsum_rows<float>((const float*)a.dye, a.expert_rows, a.db2, E, R, d, s) == cudaSuccess ? 1 : -1);
  if (a.db1) {
    if (tc)
      BW_STEP(launch_colsum_rows<__nv_bfloat16>((const __nv_bfloat16*)a.dh16, a.expert_rows, a.db1, E, R, F, s) == cudaSuccess
                  ? 1 : -1);
    else
      BW_STEP(launch_colsum_rows<float>((const float*)a.dh, a.expert_rows, a.db1, E, R, F, s) == cudaSuccess ? 1 : -1);
  }
  if (N == 0) {  // no tokens: the router's gradients are zero
    if (cudaMemsetAsync(a.dWr, 0, (size_t)E * d * sizeof(float), s) != cudaSuccess) return -1;
    if (a.dbr && cudaMemsetAsync(a.dbr, 0, (size_t)E * sizeof(float), s) != cudaSuccess) return -1;
  }
  if (N > 0) {
    const float aux_coef = a.w_aux * a.alpha * (float)E / ((float)a.G * (float)a.T * (float)a.T);  // f = raw / T
    const float z_coef = a.w_z * 2.f / ((float)a.G * (float)a.T);
    const bool tc_router = tc && a.ntc > 0;
    BW_STEP(launch_k(router_bwd_kernel, dim3((unsigned)((N + 7) / 8)), dim3(256), 0, s, false, 1, a.logits, a.expert,
                     (const float*)a.dg, a.raw, a.dz, tc_router ? (__nv_bfloat16*)a.dzp : (__nv_bfloat16*)nullptr, N, a.T, E, a.G,
                     aux_coef, z_coef) == cudaSuccess ? 1 : -1);
    if (tc_router) {
      // dWr = dz^T x on the tensor cores: token chunks of kc rows as the contraction axis,
      // dz as [hi | lo] pieces (2E output rows per chunk, x exact in bfloat16), float32
      // partials [ntc, 2E, d] summed in chunk and piece order
      split_wr3_kernel<<<592, 256, 0, s>>>(a.Wr, (__nv_bfloat16*)a.Wp, (long long)E * d);
      fill_i32_kernel<<<(a.ntc + 255) / 256, 256, 0, s>>>(a.rows_k, a.ntc, 2 * E);
      fill_i32_kernel<<<1, 32, 0, s>>>(a.rows_k + a.ntc, 1, (int)N);
      if (cudaGetLastError() != cudaSuccess) return -1;
      n += 3;
      if (cudaMemsetAsync(a.counters2, 0, (size_t)a.counter2_words * sizeof(uint32_t), s) != cudaSuccess) return -1;
      FfnLaunch M{};
      M.W1 = a.x;   // A: features c < d, rows = the chunk's tokens
      M.W2 = M.W1;
      M.xe = a.dzp; // B: the first 2E of 3E columns, rows = the chunk's tokens
      M.expert_rows = a.rows_k;
      M.mode = 2;
      M.counters = a.counters2;
      M.err = a.err;
      M.E = a.ntc;
      M.R = 2 * E;
      M.bcols = 3 * E;
      M.F = d;
      M.d = a.kc;
      M.krows = a.kc;
      M.out_f32 = a.part;
      BW_STEP(launch_ffn_tc(M, s, false));
      BW_STEP(launch_colsum_rows<float>((const float*)a.part, (const int32_t*)nullptr, a.dWr, 1, 2 * a.ntc, E * d, s) ==
                      cudaSuccess ? 1 : -1);
      // dx = dz W_r: the product over 3E of dzp [N, 3E] (K-major rows) and Wp [3E, d] (as
      // stored, MN-major), float32 results straight into dx
      if (cudaMemsetAsync(a.counters2, 0, (size_t)a.counter2_words * sizeof(uint32_t), s) != cudaSuccess) return -1;
      FfnLaunch X{};
      X.W1 = a.Wp;
      X.W2 = X.W1;
      X.xe = a.dzp;
      X.expert_rows = a.rows_k + a.ntc;
      X.mode = 3;
      X.counters = a.counters2;
      X.err = a.err;
      X.E = 1;
      X.R = (int)N;
      X.d = 3 * E;
      X.F = d;
      X.out_f32 = a.dx;
      BW_STEP(launch_ffn_tc(X, s, false));
    } else {
      // dWr = dz^T x (i = e, j = c, k = t), split over nsplit token chunks: partial results
      // per chunk, then their sum in chunk order
      const int ns = a.nsplit;
      const int kc = (int)((N + ns - 1) / ns);
      BgemmArgs g{};
      g.M = E; g.N = d; g.K = kc; g.Ktot = N;
      g.sAb = (long long)kc * E; g.sAi = 1; g.sAk = E;
      g.sBb = (long long)kc * d; g.sBj = 1; g.sBk = d;
      g.sCb = (long long)E * d; g.sCi = d; g.sCj = 1;
      BW_STEP((launch_bg<float, T, float, 0, false>(a.dz, x, a.part, nullptr, g, ns, s)));
      BW_STEP(launch_colsum_rows<float>((const float*)a.part, (const int32_t*)nullptr, a.dWr, 1, ns, E * d, s) == cudaSuccess
                  ? 1 : -1);
    }
    if (a.dbr) {  // dbr = sum_t dz_t, split over token chunks, then the chunks' sum in order
      const int ns = a.nsplit;
      const int kc = (int)((N + ns - 1) / ns);
      colsum_split_kernel<<<dim3((unsigned)((E + 255) / 256), (unsigned)ns), 256, 0, s>>>(a.dz, a.part, N, E, kc);
      if (cudaGetLastError() != cudaSuccess) return -1;
      ++n;
      BW_STEP(launch_colsum_rows<float>((const float*)a.part, (const int32_t*)nullptr, a.dbr, 1, ns, E, s) == cudaSuccess ? 1 : -1);
    }
    if (!tc_router) {  // dx = dz Wr: i = t, j = c, k = e
      BgemmArgs g{};
      g.M = (int)N; g.N = d; g.K = E;
      g.sAi = E; g.sAk = 1;
      g.sBj = 1; g.sBk = d;
      g.sCi = d; g.sCj = 1;
      BW_STEP((launch_bg<float, float, float, 0, false>(a.dz, a.Wr, a.dx, nullptr, g, 1, s)));
    }
    if (tc)
      BW_STEP(launch_k(dx_assemble_kernel<T, __nv_bfloat16>, dim3((unsigned)((N + 7) / 8)), dim3(256), 0, s, false, 1,
                       a.dx, (const __nv_bfloat16*)a.dxe16, dy, a.expert, a.row, N, d, R, a.residual ? 1 : 0) ==
                      cudaSuccess ? 1 : -1);
    else
      BW_STEP(launch_k(dx_assemble_kernel<T, float>, dim3((unsigned)((N + 7) / 8)), dim3(256), 0, s, false, 1, a.dx,
                       (const float*)a.dxe, dy, a.expert, a.row, N, d, R, a.residual ? 1 : 0) == cudaSuccess ? 1 : -1);
  }
#undef BW_STEP
  return n;
}

int launch_backward(const BackwardArgs& a, cudaStream_t s) {
  return a.bf16 ? run_backward<__nv_bfloat16>(a, s) : run_backward<float>(a, s);
}

}  // namespace smoe
