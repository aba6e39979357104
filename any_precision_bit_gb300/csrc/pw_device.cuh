// pw_device.cuh -- device helpers shared by the kernels: number formats, the m16n8k16 MMA,
// the bit-plane -> code transpose (also used by the debug read-back, so that
// pw_unpack_indices checks the forward's own extraction), and thin wrappers over the
// mbarrier / bulk-copy (TMA) / cp.async instructions of sm_90+.
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

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8x8 bit transpose inside every byte column of eight words:
// out word s, bit (8e + p) = in word p, bit (8e + s).
__device__ __forceinline__ void transpose8(uint32_t (&X)[8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t t = ((X[j] >> 4) ^ X[j + 4]) & 0x0F0F0F0Fu;
    X[j + 4] ^= t;
    X[j] ^= t << 4;
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = (jj & 1) + (jj >> 1) * 4;  // 0,1,4,5
    uint32_t t = ((X[j] >> 2) ^ X[j + 2]) & 0x33333333u;
    X[j + 2] ^= t;
    X[j] ^= t << 2;
  }
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = 2 * jj;  // 0,2,4,6
    uint32_t t = ((X[j] >> 1) ^ X[j + 1]) & 0x55555555u;
    X[j + 1] ^= t;
    X[j] ^= t << 1;
  }
}

// Codes of one thread's fragment elements for one 128-column chunk.  w[p] = the two words
// (row g, row g+8) of plane p.  Afterwards byte e of Yg[s] is the code of element (s, e)
// of row g with plane 0 in bit 7 (MSB-aligned); the Q-bit code is byte >> (8 - Q).
template <int Q>
__device__ __forceinline__ void codes_from_planes(const uint2 (&w)[Q], uint32_t (&Yg)[8],
                                                  uint32_t (&Y8)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    Yg[i] = 0u;
    Y8[i] = 0u;
  }
#pragma unroll
  for (int p = 0; p < Q; ++p) {
    Yg[7 - p] = w[p].x;
    Y8[7 - p] = w[p].y;
  }
  transpose8(Yg);
  transpose8(Y8);
}

template <int Q>
__device__ __forceinline__ uint32_t code_at(uint32_t Y, int e) {
  return (Y >> (8 * e + 8 - Q)) & ((1u << Q) - 1u);
}

// Two 16-bit shared-memory loads packed into one register (low = first address).
__device__ __forceinline__ uint32_t lds_pair(uint32_t a_lo, uint32_t a_hi) {
  uint32_t r;
  asm volatile(
      "{\n .reg .b16 lo, hi;\n ld.shared.b16 lo, [%1];\n ld.shared.b16 hi, [%2];\n"
      " mov.b32 %0, {lo, hi};\n}\n"
      : "=r"(r)
      : "r"(a_lo), "r"(a_hi));
  return r;
}
__device__ __forceinline__ void ldm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
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
// Bulk copy global -> shared through the TMA unit; completes `bytes` of the barrier's
// transaction count.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Programmatic dependent launch.  pdl_wait: block until the grids this one depends on have
// completed and their memory is visible (returns at once for a launch without a
// programmatic dependency).  pdl_trigger: let the next grid of the stream be scheduled now;
// it still waits in its own pdl_wait for this one to complete.
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
// 16-byte asynchronous copy; src_bytes = 0 fills the destination with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}
// cp.async groups: close the current group; wait until at most N of this thread's groups
// are still in flight.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace pw
