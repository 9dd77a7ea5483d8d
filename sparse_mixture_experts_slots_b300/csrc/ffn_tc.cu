// Grouped expert linear layer on 5th-generation tensor cores (tcgen05, sm_103a).
//
// One CTA computes a 128 x BN tile of   out^T[m, n] = sum_k W[e, m, k] * in[e*R + n, k]
// ("swap AB": the expert's weight rows fill the 128-row MMA; the expert's tokens,
// often only a few dozen, are the N side).  The expert FFN of the Switch layer
// is d -> d_ff, ReLU, d_ff -> d with biases ("混合专家", world.lapla.si/zh/moe,
// section 专家里面是什么); bf16 operands with f32 accumulation follow the
// bfloat16 expert computation of the Switch Transformers card (ai-papers.xuzou.cn,
// 方法适配), where only the router runs in float32.
//
// Pipeline per CTA (128 threads):
//   warp 0, one lane : TMA producer. Loads 128x64 bf16 tiles of W and BNx64 tiles
//                      of the activations (128-byte swizzle) into a STAGES-deep ring.
//   warp 1, one lane : MMA issuer. 4 x tcgen05.mma (K = 16 each) per stage into a
//                      128-lane x BN-column f32 accumulator in TMEM; tcgen05.commit
//                      frees the stage.
//   warps 0-3        : epilogue. tcgen05.ld of their 32 TMEM lanes, + bias,
//                      optional ReLU, bf16, store to out[e*R + n, m].
// Every mbarrier wait is bounded; on timeout the CTA sets the error flag, drains
// its own TMA copies and MMAs (bounded again), frees TMEM and returns.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace smoe {

constexpr int TC_BM = 128;
constexpr int TC_BK = 64;  // 64 bf16 = 128 bytes = one swizzle row

template <int BN, int STAGES>
struct TcLayout {
  static constexpr int A_BYTES = TC_BM * TC_BK * 2;
  static constexpr int B_BYTES = BN * TC_BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int SMEM_BYTES = BAR_OFFSET + 256 + 1024;  // barriers + 1024-byte alignment slack
  static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;    // power of two >= 32
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 M=128 needs N % 16 == 0, 16..256");
  static_assert((BN & (BN - 1)) == 0, "BN is a power of two here (TMEM allocation)");
};

template <int BN, int STAGES, bool RELU>
__global__ void __launch_bounds__(128, 1)
    grouped_linear_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                             const __nv_bfloat16* __restrict__ bias, __nv_bfloat16* __restrict__ out,
                             const int32_t* __restrict__ expert_rows, int R, int M, int K, uint32_t* err) {
  using L = TcLayout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * L::A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFFSET);
  uint64_t* empty = full + STAGES;
  uint64_t* accb = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int e = blockIdx.z;
  const int m0 = blockIdx.x * TC_BM;
  const int n0 = blockIdx.y * BN;
  const int rows = expert_rows[e];
  if (n0 >= rows) return;  // CTA-uniform, before any barrier or TMEM use

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int KB = K / TC_BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    const uint64_t w_policy = policy_evict_first();  // each weight tile is read by one CTA per n-tile
    int issued = 0;
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % STAGES;
      if (kb >= STAGES && !mbar_wait(&empty[s], ((kb / STAGES) - 1) & 1)) {
        raise_error(err, ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      mbar_arrive_expect_tx(&full[s], L::STAGE_BYTES);
      tma_load_2d_hint(sA + s * L::A_BYTES, &tmW, &full[s], kb * TC_BK, e * M + m0, w_policy);
      tma_load_2d(sB + s * L::B_BYTES, &tmX, &full[s], kb * TC_BK, e * R + n0);
      issued = kb + 1;
    }
    // Drain: every copy this thread started has landed before the CTA may exit.
    for (int kb = issued > STAGES ? issued - STAGES : 0; kb < issued; ++kb)
      if (!mbar_wait(&full[kb % STAGES], (kb / STAGES) & 1)) raise_error(err, ERR_TIMEOUT);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(TC_BM, BN);
    for (int kb = 0; kb < KB; ++kb) {
      const int s = kb % STAGES;
      if (!mbar_wait(&full[s], (kb / STAGES) & 1)) {
        raise_error(err, ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + s * L::A_BYTES);
      const uint32_t b0 = smem_u32(sB + s * L::B_BYTES);
#pragma unroll
      for (int k = 0; k < TC_BK / 16; ++k)  // 16 bf16 = 32 bytes per MMA step inside the swizzle row
        tc_mma_bf16(tmem, sw128_kmajor_desc(a0 + k * 32), sw128_kmajor_desc(b0 + k * 32), idesc,
                    (kb > 0 || k > 0) ? 1u : 0u);
      tc_commit(&empty[s]);
    }
    tc_commit(accb);  // arrives when every MMA issued above has completed
  }
  __syncwarp();

  // ---------------- epilogue (all 4 warps; warp w owns TMEM lanes 32w..32w+31)
  const bool acc_ok = mbar_wait(accb, 0);
  if (!acc_ok) raise_error(err, ERR_TIMEOUT);
  tc_fence_after();
  if (acc_ok && !*abort_flag) {
    const int m = m0 + warp * 32 + lane;
    const float bv = bias ? __bfloat162float(bias[(size_t)e * M + m]) : 0.f;
    __nv_bfloat16* orow = out + (size_t)e * R * M + m;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int n = n0 + c0 + j;
        if (n < rows) {
          float v = __uint_as_float(r[j]) + bv;
          if (RELU) v = fmaxf(v, 0.f);
          orow[(size_t)n * M] = __float2bfloat16_rn(v);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
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
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)TC_BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_shape_ok(int M, int K) { return M > 0 && K > 0 && M % TC_BM == 0 && K % TC_BK == 0; }

template <int BN, int STAGES, bool RELU>
static int launch_tc(const CUtensorMap& tmW, const CUtensorMap& tmX, const void* bias, void* out,
                     const int32_t* expert_rows, int E, int R, int M, int K, uint32_t* err, cudaStream_t s) {
  using L = TcLayout<BN, STAGES>;
  auto kern = grouped_linear_tc_kernel<BN, STAGES, RELU>;
  static bool attr_set = false;  // per instantiation; the attribute is per device function
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES) != cudaSuccess)
      return -1;
    attr_set = true;
  }
  dim3 grid(M / TC_BM, (R + BN - 1) / BN, E);
  kern<<<grid, 128, L::SMEM_BYTES, s>>>(tmW, tmX, (const __nv_bfloat16*)bias, (__nv_bfloat16*)out, expert_rows, R,
                                        M, K, err);
  return cudaGetLastError() == cudaSuccess ? 1 : -1;
}

int launch_grouped_linear_tc(const void* in, const void* W, const void* bias, void* out,
                             const int32_t* expert_rows, int E, int R, int M, int K, bool relu, uint32_t* err,
                             cudaStream_t s) {
  if (E == 0 || R == 0) return 0;
  if (!tc_shape_ok(M, K)) return -1;
  const int BN = R <= 32 ? 32 : R <= 64 ? 64 : R <= 128 ? 128 : 256;
  CUtensorMap tmW, tmX;
  if (!encode_bf16_2d(&tmW, W, (uint64_t)E * M, (uint64_t)K, TC_BM)) return -1;
  if (!encode_bf16_2d(&tmX, in, (uint64_t)E * R, (uint64_t)K, (uint32_t)BN)) return -1;
#define SMOE_TC(BNV, ST)                                                                                      \
  return relu ? launch_tc<BNV, ST, true>(tmW, tmX, bias, out, expert_rows, E, R, M, K, err, s)               \
              : launch_tc<BNV, ST, false>(tmW, tmX, bias, out, expert_rows, E, R, M, K, err, s)
  switch (BN) {
    case 32: SMOE_TC(32, 5);
    case 64: SMOE_TC(64, 4);
    case 128: SMOE_TC(128, 3);
    default: SMOE_TC(256, 4);
  }
#undef SMOE_TC
}

}  // namespace smoe
