// Grouped linear layer on CUDA cores (sm_103a): the float32 expert FFN, and bf16
// shapes whose widths the tensor-core kernel does not tile (d or d_ff not a
// multiple of 128).  One expert FFN is d -> d_ff, ReLU, d_ff -> d with biases
// ("混合专家", world.lapla.si/zh/moe, section 专家里面是什么).
//
// out[e*R + n, m] = act( sum_k in[e*R + n, k] * W[e, m, k] + bias[e, m] ),  n < expert_rows[e]
#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int GL_BN = 64, GL_BM = 64, GL_BK = 16;

template <typename T, bool RELU>
__global__ void __launch_bounds__(256) grouped_linear_simt_kernel(const T* __restrict__ in, const T* __restrict__ W,
                                                                  const T* __restrict__ bias, T* __restrict__ out,
                                                                  const int32_t* __restrict__ expert_rows, int R,
                                                                  int M, int K) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ float as[GL_BK][GL_BN + 4];
  __shared__ float bs[GL_BK][GL_BM + 4];
  const int e = blockIdx.z;
  const int rows = expert_rows[e];
  const int n0 = blockIdx.y * GL_BN, m0 = blockIdx.x * GL_BM;
  if (n0 >= rows) return;
  const T* A = in + (size_t)e * R * K;
  const T* B = W + (size_t)e * M * K;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += GL_BK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = threadIdx.x + 256 * i;
      const int r = idx / GL_BK, k = idx % GL_BK;
      const int n = n0 + r, m = m0 + r, kk = k0 + k;
      as[k][r] = (n < rows && kk < K) ? ld_f32(A + (size_t)n * K + kk) : 0.f;
      bs[k][r] = (m < M && kk < K) ? ld_f32(B + (size_t)m * K + kk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < GL_BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = bs[k][tx + 16 * j];
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
    if (n >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + tx + 16 * j;
      if (m >= M) continue;
      float v = acc[i][j] + (bias ? ld_f32(bias + (size_t)e * M + m) : 0.f);
      if (RELU) v = fmaxf(v, 0.f);
      out[((size_t)e * R + n) * M + m] = act_traits<T>::from_f32(v);
    }
  }
}

int launch_grouped_linear_simt(const void* in, const void* W, const void* bias, void* out,
                               const int32_t* expert_rows, int E, int R, int M, int K, bool relu, bool bf16,
                               cudaStream_t s, bool pdl) {
  if (E == 0 || R == 0) return 0;
  dim3 grid((M + GL_BM - 1) / GL_BM, (R + GL_BN - 1) / GL_BN, E);
  cudaError_t e;
#define SMOE_GL(T, RL)                                                                                           \
  e = launch_k(grouped_linear_simt_kernel<T, RL>, grid, dim3(256), 0, s, pdl, 1, (const T*)in, (const T*)W,     \
               (const T*)bias, (T*)out, expert_rows, R, M, K)
  if (bf16) {
    if (relu) SMOE_GL(__nv_bfloat16, true); else SMOE_GL(__nv_bfloat16, false);
  } else {
    if (relu) SMOE_GL(float, true); else SMOE_GL(float, false);
  }
#undef SMOE_GL
  return e == cudaSuccess ? 1 : -1;
}

}  // namespace smoe
