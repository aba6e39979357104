// pw_device.cuh -- device helpers shared by the kernels: number formats, the 8x8 bit
// transpose behind the bit-plane -> code extraction (also used by the debug read-back, so
// that pw_unpack_indices checks the forward's own extraction), thin wrappers over the
// mbarrier, bulk-copy and TMA tensor instructions, and programmatic dependent launch.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace pw {

__device__ __forceinline__ float bf16f(uint32_t b) { return __uint_as_float((b & 0xFFFFu) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) { return (lo & 0xFFFFu) | (hi << 16); }
__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// One step of a bit-matrix transpose: the bits of b under mask M trade places with the bits
// of a under M << S.  Written as two masked merges (one three-input logic operation each)
// of a with b << S and of b with a >> S, which takes fewer integer-pipe instructions than
// the usual exchange through a XOR difference.
// Shifts by a constant written as multiplies (low and high word of x * 2^s), which the
// multiply-add pipe executes, to leave the integer/logic pipe to the masked merges.
template <int S>
__device__ __forceinline__ uint32_t shl_mul(uint32_t x) {
  uint32_t r;
  asm("mul.lo.u32 %0, %1, %2;" : "=r"(r) : "r"(x), "n"(1u << S));
  return r;
}
template <int S>
__device__ __forceinline__ uint32_t shr_mul(uint32_t x) {
  uint32_t r;
  asm("mul.hi.u32 %0, %1, %2;" : "=r"(r) : "r"(x), "n"(1u << (32 - S)));
  return r;
}

template <int S, uint32_t M>
__device__ __forceinline__ void bit_swap(uint32_t &a, uint32_t &b) {
  constexpr uint32_t MH = M << S;
  const uint32_t bs = shl_mul<S>(b), as = shr_mul<S>(a);
  const uint32_t na = (a & ~MH) | (bs & MH);
  const uint32_t nb = (b & ~M) | (as & M);
  a = na;
  b = nb;
}

// 8x8 bit transpose inside every byte column of eight words:
// out word s, bit (8e + p) = in word p, bit (8e + s).
__device__ __forceinline__ void transpose8(uint32_t (&X)[8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) bit_swap<4, 0x0F0F0F0Fu>(X[j], X[j + 4]);
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = (jj & 1) + (jj >> 1) * 4;  // 0,1,4,5
    bit_swap<2, 0x33333333u>(X[j], X[j + 2]);
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = 2 * jj;  // 0,2,4,6
    bit_swap<1, 0x55555555u>(X[j], X[j + 1]);
  }
}

// ------------------------------------------------------------------ async copies, mbarriers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait with a suspend-time hint: a thread whose phase is not complete is taken off the
// scheduler until the phase completes or about `ns` nanoseconds pass, instead of spending
// issue slots on polling.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bulk copy global -> shared through the TMA unit; completes `bytes` of the barrier's
// transaction count.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// L2 cache policy for data read once (streamed weights): its lines are the first to go, so
// that what is re-read (activations, h) stays in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
  return p;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
// Programmatic dependent launch.  pdl_wait: block until the grids this one depends on have
// completed and their memory is visible (returns at once for a launch without a
// programmatic dependency).  pdl_trigger: let the next grid of the stream be scheduled now;
// it still waits in its own pdl_wait for this one to complete.
// Order this thread's generic-proxy global writes (or what it has observed of other threads')
// before later tensor-copy (async-proxy) accesses of global memory.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;\n" ::: "memory");
}
// Load with acquire semantics at GPU scope.
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Launch with programmatic stream serialisation: the kernel may be scheduled before the
// previous kernel of the stream has completed, and waits for it in pdl_wait.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}
// TMA load of one box of a 2-D tensor map (`tmap`: the map's generic address, in kernel
// parameter space) at element coordinates (x = column, y = row) into shared memory,
// completing on the mbarrier.  x times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
}  // namespace pw
