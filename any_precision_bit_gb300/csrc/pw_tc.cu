// pw_tc.cu -- self-check of the tcgen05 building blocks used by the tensor-core expert path:
// one CTA computes D[128][N] = A[128][K] * B[N][K]^T (fp16 in, fp32 out) with B in the
// core-matrix shared-memory layout of pw_tc.cuh, A either in that layout too or written into
// tensor memory with tcgen05.st (row m in lane m, K-elements 2c, 2c+1 in column c), the
// accumulator in tensor memory, the MMAs completing on an mbarrier and the result read back
// with tcgen05.ld.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw_device.cuh"
#include "pw_internal.h"
#include "pw_tc.cuh"

namespace pw {

constexpr long kTcSpin = 1L << 24;

__global__ void __launch_bounds__(128, 1) tc_selftest_kernel(const uint16_t *A, const uint16_t *B, int N, int K,
                                                             int a_tmem, float *D, int *err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  uint8_t *sa = sm;
  uint8_t *sb = sm + 128 * K * 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kc = K / 8;
  for (int i = tid; i < 128 * K; i += 128) {
    const int r = i / K, c = i % K;
    *reinterpret_cast<uint16_t *>(sa + core_offset(r, c, kc)) = A[i];
  }
  for (int i = tid; i < N * K; i += 128) {
    const int r = i / K, c = i % K;
    *reinterpret_cast<uint16_t *>(sb + core_offset(r, c, kc)) = B[i];
  }
  fence_async_smem();
  uint32_t ncols = 32;
  while ((int)ncols < N + (a_tmem ? K / 2 : 0)) ncols <<= 1;
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tslot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = tslot;
  const uint32_t acol = (uint32_t)N;  // A columns follow the accumulator's
  if (a_tmem) {  // thread = row 32 * warp + lane writes its K / 2 fp16 pairs
    const int row = 32 * warp + lane;
    for (int c0 = 0; c0 < K / 2; c0 += 16) {
      uint32_t v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int k = 2 * (c0 + i);
        v[i] = k < K ? (uint32_t)A[row * K + k] | ((uint32_t)A[row * K + k + 1] << 16) : 0u;
      }
      tmem_st16(taddr + ((uint32_t)(32 * warp) << 16) + acol + (uint32_t)c0, v);
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t idesc = idesc_f16_f32(128, N);
    const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
    for (int t = 0; t < K / 16; ++t) {
      const uint64_t bd = smem_desc(b0 + 256 * t, 128, kc * 128);
      if (a_tmem)
        tc_mma_f16_ta(taddr, taddr + acol + 8 * t, bd, idesc, t > 0 ? 1u : 0u);
      else
        tc_mma_f16(taddr, smem_desc(a0 + 256 * t, 128, kc * 128), bd, idesc, t > 0 ? 1u : 0u);
    }
    tc_commit(smem_u32(&bar));
  }
  bool ok = false;
  for (long i = 0; i < kTcSpin; ++i)
    if (mbar_try_wait(smem_u32(&bar), 0)) {
      ok = true;
      break;
    }
  tc_fence_after();
  if (!ok) {
    if (tid == 0) atomicExch(err, 1);
  } else {
    const int row = 32 * warp + lane;
    for (int c = 0; c < N; c += 16) {
      uint32_t r[16];
      tmem_ld16(taddr + ((uint32_t)(32 * warp) << 16) + (uint32_t)c, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) D[(size_t)row * N + c + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(taddr, ncols);
}

int launch_tc_selftest(const uint16_t *A, const uint16_t *B, int N, int K, int a_tmem, float *D, int *err,
                       void *stream) {
  const int smem = (128 + N) * K * 2;
  cudaFuncSetAttribute(tc_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  tc_selftest_kernel<<<1, 128, smem, reinterpret_cast<cudaStream_t>(stream)>>>(A, B, N, K, a_tmem, D, err);
  return (int)cudaGetLastError();
}

}  // namespace pw

extern "C" pw_status pw_tc_selftest(const uint16_t *A, const uint16_t *B, int N, int K, int flags, float *D,
                                    int *err, pw_stream stream) {
  if (!A || !B || !D || !err) return PW_ERR_INVALID;
  if (N < 16 || N > 256 || N % 16 || K < 16 || K > 128 || K % 16 || (flags & ~1)) return PW_ERR_INVALID;
  if (pw::launch_tc_selftest(A, B, N, K, flags & 1, D, err, stream)) return PW_ERR_CUDA;
  return PW_OK;
}
