// pw_dq.cuh -- from a row's bit-plane words to fp16 centroids (PagedWeight Sec. 3.1 weight
// pages: Any-Precision bit-planes, plane 0 the most significant, with a per-row LUT for each
// supported bitwidth).  Used by the expert kernels and by the read-back kernels, so that the
// read-back checks the very code the forward runs.
//
// Input: the Q words W[p] (plane p) of one row and one 32-column group, in the nibble-major
// bit order of the plane tiling (bit 4 i + j holds column 8 j + i).  Output: 16 registers
// v[t], t = 0..15, each the fp16 centroids of columns 2t (low half) and 2t + 1 (high half).
//   Q <= kRegLutMaxQ: a 4x4 bit transpose across the planes gives word j = the 4-bit codes of columns
//           8j..8j+7 (column 8j + i in nibble i).  The row's LUT sits in registers as the
//           low bytes and the high bytes of its centroids; byte permutes (prmt) look up four
//           codes at a time and interleave the bytes into fp16 pairs.
//   wider: an 8x8 bit transpose gives word s, byte e = the code of column
//           8 (s & 3) + 2e + (s >> 2).  The LUT is in shared memory in the tiled layout of
//           lut_dev_index (pw_internal.h): the code is byte 1 of its entry's address, so one
//           byte permute forms the address, every lane of a warp reads its own bank, and two
//           16-bit loads joined by a multiply-add give each pair.
// The decode keeps the integer/logic pipe busiest (it issues at half the rate of the
// multiply-add pipe), so the steps are chosen to spend as few of its instructions as they
// can: masked-merge transposes, no separate step for the table's address bits, and the
// pairs joined on the multiply-add pipe.
#pragma once
#include <stdint.h>

#include "pw_device.cuh"

namespace pw {

// Widths up to this one look centroids up in registers (byte permutes); wider ones in the
// shared-memory LUT.  At 4 bits the shared-memory path is the faster one: the register path
// needs a second level of permutes to pick between two 8-entry halves.
#ifndef PW_REG_LUT_MAX_Q
#define PW_REG_LUT_MAX_Q 3
#endif
constexpr int kRegLutMaxQ = PW_REG_LUT_MAX_Q;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 4x4 bit transpose inside every nibble column of four words:
// out word s, bit (4i + p) = in word p, bit (4i + s).
__device__ __forceinline__ void transpose4(uint32_t (&X)[4]) {
#pragma unroll
  for (int j = 0; j < 2; ++j) bit_swap<2, 0x33333333u>(X[j], X[j + 2]);
#pragma unroll
  for (int j = 0; j < 4; j += 2) bit_swap<1, 0x55555555u>(X[j], X[j + 1]);
}

// A LUT of up to 16 centroids as byte planes: lo[m] byte b = low byte of entry 4m + b,
// hi[m] likewise for the high bytes.
struct LutRegs {
  uint32_t lo[4], hi[4];
};
// From the entries as fp16 pairs P[i] = entry 2i | entry 2i+1 << 16 (unused entries zero).
__device__ __forceinline__ void lut_regs(const uint32_t (&P)[8], LutRegs &L) {
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    L.lo[m] = prmt(P[2 * m], P[2 * m + 1], 0x6420);
    L.hi[m] = prmt(P[2 * m], P[2 * m + 1], 0x7531);
  }
}

// Q <= 4: codes of the 32 columns, word j = columns 8j..8j+7 (nibble i = column 8j + i).
template <int Q>
__device__ __forceinline__ void codes_nib(const uint32_t (&W)[8], uint32_t (&S)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) S[i] = 0u;
#pragma unroll
  for (int p = 0; p < Q; ++p) S[Q - 1 - p] = W[p];
  transpose4(S);
}

// Q <= 4: centroids of four codes (the low 16 bits of s hold them, one per nibble), as the
// low bytes and the high bytes of the four results.
template <int Q>
__device__ __forceinline__ void lut4(uint32_t s, const LutRegs &L, uint32_t &lo, uint32_t &hi) {
  if constexpr (Q <= 3) {
    lo = prmt(L.lo[0], L.lo[1], s);
    hi = prmt(L.hi[0], L.hi[1], s);
  } else {
    // prmt reads nibble bit 3 as a sign-replicate flag: look up with bits 0..2 in both
    // halves of the table, then pick per byte by bit 3
    const uint32_t s7 = s & 0x7777u;
    const uint32_t sel = ((s >> 1) & 0x4444u) | 0x3210u;
    lo = prmt(prmt(L.lo[0], L.lo[1], s7), prmt(L.lo[2], L.lo[3], s7), sel);
    hi = prmt(prmt(L.hi[0], L.hi[1], s7), prmt(L.hi[2], L.hi[3], s7), sel);
  }
}

template <int Q>
__device__ __forceinline__ void dq_nib(const uint32_t (&S)[4], const LutRegs &L, uint32_t (&v)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t lo, hi;
      lut4<Q>(h ? (S[j] >> 16) : S[j], L, lo, hi);
      v[4 * j + 2 * h] = prmt(lo, hi, 0x5140);
      v[4 * j + 2 * h + 1] = prmt(lo, hi, 0x7362);
    }
  }
}

// Q >= 4 (any Q works): codes of the 32 columns, word s byte e = code of column
// 8 (s & 3) + 2e + (s >> 2), plane 0 in bit Q - 1 (the byte is the code itself).  For Q <= 7
// bit 7 of every byte is bit 7 of `top` (0 or ~0): the shared-memory LUT addressing below
// uses it for the table's address bit 15.
template <int Q>
__device__ __forceinline__ void codes_byte(const uint32_t (&W)[8], uint32_t (&Y)[8], uint32_t top = 0u) {
#pragma unroll
  for (int i = 0; i < 8; ++i) Y[i] = 0u;
  if constexpr (Q < 8) Y[7] = top;
#pragma unroll
  for (int p = 0; p < Q; ++p) Y[Q - 1 - p] = W[p];
  transpose8(Y);
}

// Shared-memory LUT of the tiled layout (lut_dev_index) as seen by one lane: `word0` is the
// address of the lane's word for code 0 (table base + 128 (m >> 1) + 4 L for lane quarter m,
// lane L; the table base is 64 KB-aligned, or 32 KB past that for a table of at most 128
// codes), `half` selects the lane's row in each word (0x5410: low halves, 0x7632: high),
// `h16` is the address of the lane's own 16-bit centroid of code 0 and `top` the word that
// codes_byte needs for the table's address bit 15.
struct LutLane {
  uint32_t word0, half, h16, top;
};
__device__ __forceinline__ LutLane lut_lane(uint32_t table, int quarter, int lane) {
  const uint32_t w0 = table + 128u * (uint32_t)(quarter >> 1) + 4u * (uint32_t)lane;
  return LutLane{w0, (quarter & 1) ? 0x7632u : 0x5410u, w0 + 2u * (uint32_t)(quarter & 1),
                 (table & 0x8000u) ? 0xFFFFFFFFu : 0u};
}
__device__ __forceinline__ uint32_t lds_b32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}
// lo | hi << 16 for 16-bit lo and hi, as a multiply-add (the multiply-add pipe is idle while
// the decode keeps the integer pipe busy)
__device__ __forceinline__ uint32_t pack_mad(uint32_t lo, uint32_t hi) {
  uint32_t v;
  asm("mad.lo.u32 %0, %1, 65536, %2;" : "=r"(v) : "r"(hi), "r"(lo));
  return v;
}

// Q <= 4: the lane's row of LUT_Q from shared memory as fp16 pairs P[i] = entries 2i, 2i+1.
template <int Q>
__device__ __forceinline__ void lut_pairs_smem(const LutLane &lu, uint32_t (&P)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    P[i] = 0u;
    if (2 * i + 1 < (1 << Q))
      P[i] = prmt(lds_b32(lu.word0 + 512u * i), lds_b32(lu.word0 + 512u * i + 256u), lu.half);
  }
}

// Q >= 4: centroids from the lane's LUT in shared memory.  The code is byte 1 of its entry's
// address (codes_byte put the table's address bit 15 into bit 7 of each code byte), so one
// byte permute with the lane's address forms it; two 16-bit loads and a multiply-add make
// the pair.
template <int Q>
__device__ __forceinline__ void dq_byte(const uint32_t (&Y)[8], const LutLane &lu, uint32_t (&v)[16]) {
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t lo = lds_u16(prmt(Y[s], lu.h16, 0x7604u | ((uint32_t)e << 4)));
      const uint32_t hi = lds_u16(prmt(Y[s + 4], lu.h16, 0x7604u | ((uint32_t)e << 4)));
      v[4 * s + e] = pack_mad(lo, hi);
    }
}

// code of column c (0..31) of the group, from the outputs of codes_nib / codes_byte
template <int Q>
__device__ __forceinline__ uint32_t code_nib(const uint32_t (&S)[4], int c) {
  return (S[c >> 3] >> (4 * (c & 7))) & 0xFu;
}
template <int Q>
__device__ __forceinline__ uint32_t code_byte(const uint32_t (&Y)[8], int c) {
  const int j = c >> 3, i = c & 7;  // column 8j + i = 8 (s & 3) + 2e + (s >> 2)
  const int s = j + 4 * (i & 1), e = i >> 1;
  return (Y[s] >> (8 * e)) & ((1u << Q) - 1u);
}

}  // namespace pw
