// pw_kernels.cu -- decode-path kernels of the fused mixed-precision MoE layer (sm_103a).
//
// PagedWeight Sec. 3.3 ("Fused Mixed-Precision MoE Kernel"): routing, expert activation,
// down projection and output accumulation, each linear block read directly from its AP
// bit-planes and LUT at its committed bitwidth.  Here one layer is four launches:
//   route_kernel   router logits (fp32), softmax, top-K; the last CTA to finish buckets
//                  the (token, k) pairs by expert and writes the work lists
//   ffn_kernel<1>  gate_up of every active expert and of the shared expert, SiLU(g)*u
//   ffn_kernel<2>  down projection of every active expert and of the shared expert
//   combine_kernel y_t = sum_k r_tk o_tk (k order) + shared (+ y when accumulating)
//
// Expert kernels: each warp owns a 16-row tile of a block and streams its bit-planes in
// 128-column chunks.  A chunk gives every thread one 32-bit word per plane per row (the
// kernel-private tiling in pw_internal.h), which an 8x8 bit transpose turns into the
// MSB-aligned codes of exactly the elements of its m16n8k16 A fragment; the codes index
// the row's LUT_q staged in shared memory, and the fp16 centroids go straight into the
// A fragment registers.  Tokens form the N side (8 per MMA, up to 64 per work item), so
// each dequantised element is used by every token of the expert without a trip through
// shared memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw_internal.h"

namespace pw {

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ uint16_t f2h(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }
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
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
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

// ------------------------------------------------------------------ router
constexpr int kRtTok = 8;   // tokens per router CTA
constexpr int kRtExp = 8;   // experts per router CTA (one per warp)
constexpr int kRtThreads = 256;

__global__ void __launch_bounds__(kRtThreads) route_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);  // [kRtTok][H] bf16
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kRtTok;
  const int nt = min(kRtTok, a.T - t0);
  const int H = a.H, E = a.E, K = a.K;

  for (int v = tid; v < kRtTok * H / 8; v += kRtThreads) {
    int t = v / (H / 8), c = (v % (H / 8)) * 8;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (t < nt) val = *reinterpret_cast<const uint4 *>(a.x + (size_t)(t0 + t) * H + c);
    *reinterpret_cast<uint4 *>(xs + t * H + c) = val;
  }
  __syncthreads();
  // unit-gain RMSNorm of the layer input (PW_PRENORM): one warp per staged token
  __shared__ float s_inv[kRtTok];
  if (warp < kRtTok) {
    float ss = 0.f;
    for (int h = lane * 2; h < H; h += 64) {
      const uint32_t v = *reinterpret_cast<const uint32_t *>(xs + warp * H + h);
      const float a0 = bf16f(v & 0xFFFF), a1 = bf16f(v >> 16);
      ss = fmaf(a0, a0, fmaf(a1, a1, ss));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = (a.flags & 2) ? rsqrtf(ss / (float)H + 1e-6f) : 1.0f;
    if (lane == 0) {
      s_inv[warp] = inv;
      if (blockIdx.y == 0 && warp < nt) a.s.inv_rms[t0 + warp] = inv;
    }
  }
  __syncthreads();
  const int e = blockIdx.y * kRtExp + warp;
  if (e < E) {
    float acc[kRtTok];
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) acc[t] = 0.f;
    const float *wr = a.lay.Wr + (size_t)e * H;
    for (int h = lane * 4; h < H; h += 128) {
      float4 wv = *reinterpret_cast<const float4 *>(wr + h);
#pragma unroll
      for (int t = 0; t < kRtTok; ++t) {
        uint2 xv = *reinterpret_cast<const uint2 *>(xs + t * H + h);
        acc[t] = fmaf(bf16f(xv.x & 0xFFFF), wv.x, acc[t]);
        acc[t] = fmaf(bf16f(xv.x >> 16), wv.y, acc[t]);
        acc[t] = fmaf(bf16f(xv.y & 0xFFFF), wv.z, acc[t]);
        acc[t] = fmaf(bf16f(xv.y >> 16), wv.w, acc[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t < nt) {
        float b = a.lay.bias ? a.lay.bias[e] : 0.f;
        a.s.logits[(size_t)(t0 + t) * E + e] = v * s_inv[t] + b;
      }
    }
  }

  // ---- the last CTA to finish runs the per-layer global part
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    unsigned total = gridDim.x * gridDim.y;
    unsigned old = atomicAdd(a.s.ticket, 1u);
    s_last = (old == total - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int T = a.T, TK = a.T * a.K;
  // softmax + top-K, one warp per token
  for (int t = warp; t < T; t += kRtThreads / 32) {
    const float *lg = a.s.logits + (size_t)t * E;  // written by other CTAs: read through L2
    float lv[8];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int ee = lane + 32 * i;
      lv[i] = (ee < E) ? __ldcg(lg + ee) : -INFINITY;
      mx = fmaxf(mx, lv[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int ee = lane + 32 * i;
      lv[i] = (ee < E) ? expf(lv[i] - mx) : 0.f;
      sum += lv[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = 1.0f / sum;
    unsigned taken = 0u;
    float chosen_sum = 0.f;
    float wk[8];
    int ik[8];
    for (int k = 0; k < K; ++k) {
      // a NaN probability ranks below every number, and some untaken expert always wins,
      // so the ids stay in range whatever the logits hold
      float best = -2.f;
      int bid = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int ee = lane + 32 * i;
        if (ee < E && !((taken >> i) & 1u)) {
          float p = lv[i] * inv;
          float key = (p == p) ? p : -1.f;
          if (key > best || (key == best && ee < bid)) {
            best = key;
            bid = ee;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ob = __shfl_xor_sync(0xffffffffu, best, o);
        int oi = __shfl_xor_sync(0xffffffffu, bid, o);
        if (ob > best || (ob == best && oi < bid)) {
          best = ob;
          bid = oi;
        }
      }
      bid = min(bid, E - 1);
      if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
      wk[k] = best;
      ik[k] = bid;
      chosen_sum += best;
    }
    if (lane < K) {
      float wv = 0.f;
      int iv = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (k == lane) {
          wv = wk[k];
          iv = ik[k];
        }
      if (a.renorm) wv = wv / chosen_sum;
      a.s.ids[t * K + lane] = iv;
      a.s.w[t * K + lane] = wv;
      if (a.ids_out) a.ids_out[t * K + lane] = iv;
      if (a.w_out) a.w_out[t * K + lane] = wv;
    }
  }
  __syncthreads();

  // bucketing: histogram, exclusive scan, stable (expert, token) order
  __shared__ int s_cnt[256];
  __shared__ int s_off[257];
  __shared__ int s_cur[256];
  __shared__ int s_itm1[257];
  __shared__ int s_itm2[257];
  for (int i = tid; i < 256; i += kRtThreads) s_cnt[i] = 0;
  __syncthreads();
  for (int j = tid; j < TK; j += kRtThreads) atomicAdd(&s_cnt[a.s.ids[j]], 1);
  __syncthreads();
  const int tiles1 = (2 * a.I + kCtaRows - 1) / kCtaRows;
  const int tiles2 = (a.H + kCtaRows - 1) / kCtaRows;
  const int tchunks = (T + kTokChunk - 1) / kTokChunk;
  const int sh1 = a.Is > 0 ? ((2 * a.Is + kCtaRows - 1) / kCtaRows) * tchunks : 0;
  const int sh2 = a.Is > 0 ? tiles2 * tchunks : 0;
  if (tid == 0) {
    int o = 0, i1 = sh1, i2 = sh2;
    for (int ee = 0; ee < E; ++ee) {
      s_off[ee] = o;
      s_cur[ee] = o;
      s_itm1[ee] = i1;
      s_itm2[ee] = i2;
      int ch = (s_cnt[ee] + kTokChunk - 1) / kTokChunk;
      o += s_cnt[ee];
      i1 += ch * tiles1;
      i2 += ch * tiles2;
    }
    s_off[E] = o;
    s_itm1[E] = i1;
    s_itm2[E] = i2;
    a.s.n_items[0] = i1;
    a.s.n_items[1] = i2;
  }
  __syncthreads();
  for (int i = tid; i <= E; i += kRtThreads) a.s.offsets[i] = s_off[i];
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    for (int base = 0; base < TK; base += 32) {
      int j = base + lane;
      int ee = (j < TK) ? a.s.ids[j] : -1 - lane;  // invalid lanes never match a valid one
      unsigned peers = __match_any_sync(0xffffffffu, ee);
      int rank = __popc(peers & lt);
      int leader = __ffs(peers) - 1;
      int slot = 0;
      if (j < TK) slot = s_cur[ee] + rank;
      __syncwarp();
      if (j < TK && lane == leader) s_cur[ee] += __popc(peers);
      __syncwarp();
      if (j < TK) {
        a.s.slot_tok[slot] = j / K;
        a.s.pair_slot[j] = slot;
        a.s.slot_w[slot] = a.s.w[j];
      }
    }
  }
  // shared-expert work items (first, they are the heaviest)
  for (int i = tid; i < sh1; i += kRtThreads) {
    int tile = i / tchunks, ch = i % tchunks;
    a.s.items1[i] = WorkItem{1, 0, tile, ch * kTokChunk, min(kTokChunk, T - ch * kTokChunk)};
  }
  for (int i = tid; i < sh2; i += kRtThreads) {
    int tile = i / tchunks, ch = i % tchunks;
    a.s.items2[i] = WorkItem{1, 0, tile, ch * kTokChunk, min(kTokChunk, T - ch * kTokChunk)};
  }
  __syncthreads();
  // routed work items and routing statistics, one thread per expert
  for (int ee = tid; ee < E; ee += kRtThreads) {
    const int cnt = s_cnt[ee];
    const int ch = (cnt + kTokChunk - 1) / kTokChunk;
    int p1 = s_itm1[ee], p2 = s_itm2[ee];
    for (int c = 0; c < ch; ++c) {
      int nt2 = min(kTokChunk, cnt - c * kTokChunk);
      for (int tile = 0; tile < tiles1; ++tile) a.s.items1[p1++] = WorkItem{0, ee, tile, c * kTokChunk, nt2};
      for (int tile = 0; tile < tiles2; ++tile) a.s.items2[p2++] = WorkItem{0, ee, tile, c * kTokChunk, nt2};
    }
    double ws = 0.0;
    for (int sl = s_off[ee]; sl < s_off[ee] + cnt; ++sl) ws += (double)a.s.slot_w[sl];
    a.s.stat_count[(size_t)a.layer * E + ee] += (double)cnt;
    a.s.stat_wsum[(size_t)a.layer * E + ee] += ws;
  }
  if (tid == 0) *a.s.ticket = 0u;
}

// ------------------------------------------------------------------ expert kernels
constexpr int kFfnThreads = 32 * kWarpsPerCta;
constexpr int kXCols = 512;           // activation columns staged per pass
constexpr int kXStride = kXCols + 8;  // fp16 units; +16 B keeps B-fragment reads conflict-free

struct FfnSmem {
  uint16_t *lut;  // [kCtaRows][2^q]
  uint16_t *xs;   // [xt][kXStride]
};

// Stage activation columns [c0, c0 + kXCols) of the item's tokens into xs (zero padded),
// as fp16: PHASE 1 converts the bf16 layer input (times 1/rms under PW_PRENORM) -- routed
// items gather their tokens, shared items take them in order; PHASE 2 copies the fp16 h
// rows.
template <int PHASE, bool SHARED>
__device__ __forceinline__ void stage_x(const FwdArgs &a, const WorkItem &w, int slot0, int Kc,
                                        int c0, int xt, uint16_t *xs) {
  const int vecs = kXCols / 8;
  for (int v = threadIdx.x; v < xt * vecs; v += kFfnThreads) {
    const int j = v / vecs, c = c0 + (v % vecs) * 8;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (j < w.ntok && c < Kc) {
      if (PHASE == 2 && SHARED) {
        val = *reinterpret_cast<const uint4 *>(a.s.h_shared + (size_t)(w.tok0 + j) * a.Is + c);
      } else if (PHASE == 1) {
        const int t = SHARED ? w.tok0 + j : a.s.slot_tok[slot0 + j];
        const float inv = (a.flags & 2) ? a.s.inv_rms[t] : 1.0f;
        uint4 raw = *reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + c);
        uint32_t r[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o[i] = pack2(f2h(bf16f(r[i] & 0xFFFF) * inv), f2h(bf16f(r[i] >> 16) * inv));
        val = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        val = *reinterpret_cast<const uint4 *>(a.s.h_routed + (size_t)(slot0 + j) * a.I + c);
      }
    }
    *reinterpret_cast<uint4 *>(xs + j * kXStride + (v % vecs) * 8) = val;
  }
}

// Write a finished tile: PHASE 1 -> h = silu(gate) * up for feature f; PHASE 2 -> o rows.
template <int PHASE, bool SHARED>
__device__ __forceinline__ void epilogue(const FwdArgs &a, const WorkItem &w, int slot0, int rt,
                                         int ngroups, float (&acc)[8][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= ngroups) break;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int tj = 8 * j + 2 * c + h;
      if (tj >= w.ntok) continue;
      if (PHASE == 1) {
        const int f = rt * 8 + g;
        const float hv = silu(acc[j][h]) * acc[j][2 + h];
        if (SHARED)
          a.s.h_shared[(size_t)(w.tok0 + tj) * a.Is + f] = f2h(hv);
        else
          a.s.h_routed[(size_t)(slot0 + tj) * a.I + f] = f2h(hv);
      } else {
        const int r0 = rt * 16 + g;
        float *dst = SHARED ? a.s.o_shared + (size_t)(w.tok0 + tj) * a.H
                            : a.s.o_routed + (size_t)(slot0 + tj) * a.H;
        dst[r0] = acc[j][h];
        dst[r0 + 8] = acc[j][2 + h];
      }
    }
  }
}

// Routed item at compile-time bitwidth Q.
template <int PHASE, int Q>
__device__ void routed_item(const FwdArgs &a, const WorkItem &w, const BlockDev &bd, uint8_t *smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int N = bd.N, Kc = bd.K, KC = bd.KC;
  const int d0 = w.tile * kCtaRows;
  const int rows = min(kCtaRows, N - d0);
  const int rt = w.tile * kWarpsPerCta + warp;
  const bool active = warp * kTileRows < rows;
  const int slot0 = a.s.offsets[w.expert] + w.tok0;
  const int ngroups = (w.ntok + 7) / 8;
  const int xt = ngroups * 8;

  uint16_t *lut = reinterpret_cast<uint16_t *>(smem);
  uint16_t *xs = lut + kCtaRows * (1 << Q);
  {  // stage the tile's LUT_Q rows
    const uint4 *src = reinterpret_cast<const uint4 *>(bd.lut[Q] + (size_t)d0 * (1 << Q));
    uint4 *dst = reinterpret_cast<uint4 *>(lut);
    const int nv = rows * (1 << Q) / 8;
    for (int v = threadIdx.x; v < nv; v += kFfnThreads) dst[v] = src[v];
  }
  const uint16_t *lg = lut + (warp * kTileRows + g) * (1 << Q);
  const uint16_t *l8 = lg + 8 * (1 << Q);

  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;

  const int KP = KC * kChunkCols;
  for (int c0 = 0; c0 < KP; c0 += kXCols) {
    __syncthreads();
    stage_x<PHASE, false>(a, w, slot0, Kc, c0, xt, xs);
    __syncthreads();
    if (!active) continue;
    const int kc_end = min(KC, (c0 + kXCols) / kChunkCols);
    for (int kc = c0 / kChunkCols; kc < kc_end; ++kc) {
      uint2 pw_[Q];
#pragma unroll
      for (int p = 0; p < Q; ++p)
        pw_[p] = reinterpret_cast<const uint2 *>(bd.plane[p])[(size_t)(rt * KC + kc) * 32 + lane];
      uint32_t Yg[8], Y8[8];
      codes_from_planes<Q>(pw_, Yg, Y8);
      const uint16_t *xrow = xs + g * kXStride + (kc * kChunkCols - c0) + 2 * c;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint32_t a0 = pack2(lg[code_at<Q>(Yg[s], 0)], lg[code_at<Q>(Yg[s], 1)]);
        const uint32_t a1 = pack2(l8[code_at<Q>(Y8[s], 0)], l8[code_at<Q>(Y8[s], 1)]);
        const uint32_t a2 = pack2(lg[code_at<Q>(Yg[s], 2)], lg[code_at<Q>(Yg[s], 3)]);
        const uint32_t a3 = pack2(l8[code_at<Q>(Y8[s], 2)], l8[code_at<Q>(Y8[s], 3)]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j >= ngroups) break;
          const uint16_t *xb = xrow + j * 8 * kXStride + 16 * s;
          const uint32_t b0 = *reinterpret_cast<const uint32_t *>(xb);
          const uint32_t b1 = *reinterpret_cast<const uint32_t *>(xb + 8);
          mma_f16(acc[j], a0, a1, a2, a3, b0, b1);
        }
      }
    }
  }
  if (active) epilogue<PHASE, false>(a, w, slot0, rt, ngroups, acc);
}

// Shared-expert item: dense weights (bf16 converted to fp16 when set) in the frag16 layout.
template <int PHASE>
__device__ void shared_item(const FwdArgs &a, const WorkItem &w, uint8_t *smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int N = (PHASE == 1) ? 2 * a.Is : a.H;
  const int Kc = (PHASE == 1) ? a.H : a.Is;
  const uint16_t *W = (PHASE == 1) ? a.lay.wgu : a.lay.wd;
  const int d0 = w.tile * kCtaRows;
  const int rows = min(kCtaRows, N - d0);
  const int rt = w.tile * kWarpsPerCta + warp;
  const bool active = warp * kTileRows < rows;
  const int ngroups = (w.ntok + 7) / 8;
  const int xt = ngroups * 8;
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem);
  const uint4 *Wf = reinterpret_cast<const uint4 *>(W);
  const int KS = Kc / 16;

  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;

  for (int c0 = 0; c0 < Kc; c0 += kXCols) {
    __syncthreads();
    stage_x<PHASE, true>(a, w, 0, Kc, c0, xt, xs);
    __syncthreads();
    if (!active) continue;
    const int st_end = min(KS, (c0 + kXCols) / 16);
    const uint16_t *xrow = xs + g * kXStride + 2 * c;
    for (int st = c0 / 16; st < st_end; ++st) {
      const uint4 af = Wf[(size_t)(rt * KS + st) * 32 + lane];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= ngroups) break;
        const uint16_t *xb = xrow + j * 8 * kXStride + (st * 16 - c0);
        const uint32_t b0 = *reinterpret_cast<const uint32_t *>(xb);
        const uint32_t b1 = *reinterpret_cast<const uint32_t *>(xb + 8);
        mma_f16(acc[j], af.x, af.y, af.z, af.w, b0, b1);
      }
    }
  }
  if (active) epilogue<PHASE, true>(a, w, 0, rt, ngroups, acc);
}

template <int PHASE>
__global__ void __launch_bounds__(kFfnThreads) ffn_kernel(FwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int n_items = a.s.n_items[PHASE - 1];
  const WorkItem *items = (PHASE == 1) ? a.s.items1 : a.s.items2;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const WorkItem w = items[it];
    if (w.kind == 1) {
      shared_item<PHASE>(a, w, smem_raw);
    } else {
      const int block = (a.layer * a.E + w.expert) * 2 + (PHASE - 1);
      const BlockDev &bd = a.table[block];
      switch (bd.q) {
        case 1: routed_item<PHASE, 1>(a, w, bd, smem_raw); break;
        case 2: routed_item<PHASE, 2>(a, w, bd, smem_raw); break;
        case 3: routed_item<PHASE, 3>(a, w, bd, smem_raw); break;
        case 4: routed_item<PHASE, 4>(a, w, bd, smem_raw); break;
        case 5: routed_item<PHASE, 5>(a, w, bd, smem_raw); break;
        case 6: routed_item<PHASE, 6>(a, w, bd, smem_raw); break;
        case 7: routed_item<PHASE, 7>(a, w, bd, smem_raw); break;
        default: routed_item<PHASE, 8>(a, w, bd, smem_raw); break;
      }
    }
    __syncthreads();  // the next item restages the LUT and activations in shared memory
  }
}

// ------------------------------------------------------------------ combine
__global__ void __launch_bounds__(256) combine_kernel(FwdArgs a) {
  const int t = blockIdx.x;
  const int H = a.H, K = a.K;
  __shared__ int s_slot[8];
  __shared__ float s_w[8];
  if (threadIdx.x < K) {
    s_slot[threadIdx.x] = a.s.pair_slot[t * K + threadIdx.x];
    s_w[threadIdx.x] = a.s.w[t * K + threadIdx.x];
  }
  __syncthreads();
  for (int h = threadIdx.x * 4; h < H; h += 256 * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      const float4 o = *reinterpret_cast<const float4 *>(a.s.o_routed + (size_t)s_slot[k] * H + h);
      const float r = s_w[k];
      acc.x = fmaf(r, o.x, acc.x);
      acc.y = fmaf(r, o.y, acc.y);
      acc.z = fmaf(r, o.z, acc.z);
      acc.w = fmaf(r, o.w, acc.w);
    }
    if (a.Is > 0) {
      const float4 sv = *reinterpret_cast<const float4 *>(a.s.o_shared + (size_t)t * H + h);
      acc.x += sv.x;
      acc.y += sv.y;
      acc.z += sv.z;
      acc.w += sv.w;
    }
    uint2 *yp = reinterpret_cast<uint2 *>(a.y + (size_t)t * H + h);
    if (a.flags & 1) {
      const uint2 old = *yp;
      acc.x += bf16f(old.x & 0xFFFF);
      acc.y += bf16f(old.x >> 16);
      acc.z += bf16f(old.y & 0xFFFF);
      acc.w += bf16f(old.y >> 16);
    }
    *yp = make_uint2(pack2(f2bf(acc.x), f2bf(acc.y)), pack2(f2bf(acc.z), f2bf(acc.w)));
  }
}

// ------------------------------------------------------------------ launch
static int g_smem_attr_done = -1;

static size_t ffn_smem_bytes(int xt) {
  return (size_t)kCtaRows * 256 * 2 + (size_t)xt * kXStride * 2;
}

// Timing events: under stream capture an ordinary record only orders graph nodes, so the
// record is made an external event node that fires on every replay.
static void record(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}

int launch_forward(const FwdArgs &a, void *stream_, void *const *ev_) {
  cudaEvent_t const *ev = reinterpret_cast<cudaEvent_t const *>(ev_);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  int dev = 0;
  cudaGetDevice(&dev);
  const int xt = ((min(a.T, kTokChunk) + 7) / 8) * 8;
  const size_t smem_ffn = ffn_smem_bytes(kTokChunk);  // attribute set once for the maximum
  if (g_smem_attr_done != dev) {
    cudaFuncSetAttribute(ffn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_ffn);
    cudaFuncSetAttribute(ffn_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_ffn);
    cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtTok * 8192 * 2);
    g_smem_attr_done = dev;
  }
  dim3 rg((a.T + kRtTok - 1) / kRtTok, (a.E + kRtExp - 1) / kRtExp);
  if (ev) record(ev[0], st);
  route_kernel<<<rg, kRtThreads, kRtTok * a.H * 2, st>>>(a);
  if (ev) record(ev[1], st);
  const size_t smem = ffn_smem_bytes(xt);
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ffn_kernel<1>, kFfnThreads, smem);
  if (per_sm < 1) per_sm = 1;
  const int grid1 = min(a.s.max_items1, a.sm_count * per_sm);
  const int grid2 = min(a.s.max_items2, a.sm_count * per_sm);
  ffn_kernel<1><<<grid1, kFfnThreads, smem, st>>>(a);
  if (ev) record(ev[2], st);
  ffn_kernel<2><<<grid2, kFfnThreads, smem, st>>>(a);
  if (ev) record(ev[3], st);
  combine_kernel<<<a.T, 256, 0, st>>>(a);
  if (ev) record(ev[4], st);
  return (int)cudaGetLastError();
}

// ------------------------------------------------------------------ page table / packing
__global__ void commit_kernel(BlockDev *table, int block, BlockDev val) {
  if (threadIdx.x == 0 && blockIdx.x == 0) table[block] = val;
}

int launch_commit(BlockDev *table, int block, const BlockDev &val, void *stream) {
  commit_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(table, block, val);
  return (int)cudaGetLastError();
}

// One thread per tiled word position; writes that word of every plane.
__global__ void pack_kernel(const uint8_t *idx, int N, int K, int KC, int u, int I, int bmax,
                            uint32_t *const *planes, long nwords) {
  long widx = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (widx >= nwords) return;
  const int r = (int)(widx & 1);
  const int lane = (int)((widx >> 1) & 31);
  const long tk = widx >> 6;
  const int kc = (int)(tk % KC);
  const int rt = (int)(tk / KC);
  const int g = lane >> 2, c = lane & 3;
  const int d = rt * 16 + g + 8 * r;
  const int row = orig_row(d, u, I);
  uint32_t words[kMaxPlanes] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int e = 0; e < 4; ++e) {
    const int kofs = 2 * c + (e & 1) + 8 * (e >> 1);
    for (int s = 0; s < 8; ++s) {
      const int col = kc * 128 + 16 * s + kofs;
      const uint32_t code = (col < K) ? idx[(size_t)row * K + col] : 0u;
      for (int p = 0; p < bmax; ++p) words[p] |= ((code >> (bmax - 1 - p)) & 1u) << (8 * e + s);
    }
  }
  for (int p = 0; p < bmax; ++p) planes[p][widx] = words[p];
}

int launch_pack(const uint8_t *idx, int N, int K, int KC, int u, int I, int bmax,
                uint32_t *const *plane_out, void *stream) {
  const long nwords = (long)N * KC * 4;  // N/16 tiles * KC chunks * 64 words
  const int thr = 256;
  const long blocks = (nwords + thr - 1) / thr;
  pack_kernel<<<(unsigned)blocks, thr, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      idx, N, K, KC, u, I, bmax, plane_out, nwords);
  return (int)cudaGetLastError();
}

__global__ void lut_permute_kernel(const uint16_t *in, int N, int entries, int u, int I, uint16_t *out) {
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)N * entries) return;
  const int d = (int)(i / entries), c = (int)(i % entries);
  out[i] = in[(size_t)orig_row(d, u, I) * entries + c];
}

int launch_lut_permute(const uint16_t *lut_in, int N, int entries, int u, int I, uint16_t *lut_out,
                       void *stream) {
  const long n = (long)N * entries;
  lut_permute_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      lut_in, N, entries, u, I, lut_out);
  return (int)cudaGetLastError();
}

// bf16 -> fp16 in the frag16 layout; counts values that overflow fp16 into *bad.
__global__ void frag16_kernel(const uint16_t *in, int N, int K, int u, int I, uint16_t *out, int *bad) {
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)N * K) return;
  const int d = (int)(i / K), k = (int)(i % K);
  const float v = bf16f(in[(size_t)orig_row(d, u, I) * K + k]);
  if (!(fabsf(v) <= 65504.0f)) atomicAdd(bad, 1);
  out[frag16_index(d, k, K)] = f2h(v);
}

int launch_frag16(const uint16_t *w_in, int N, int K, int u, int I, uint16_t *w_out, int *bad, void *stream) {
  const long n = (long)N * K;
  frag16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      w_in, N, K, u, I, w_out, bad);
  return (int)cudaGetLastError();
}

// Debug read-back through the forward's extraction code: one warp per (tile, chunk).
template <int Q>
__device__ void unpack_chunk(const BlockDev &bd, int rt, int kc, int u, int I, uint8_t *idx_out,
                             uint16_t *w_out) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  uint2 pw_[Q];
#pragma unroll
  for (int p = 0; p < Q; ++p)
    pw_[p] = reinterpret_cast<const uint2 *>(bd.plane[p])[(size_t)(rt * bd.KC + kc) * 32 + lane];
  uint32_t Yg[8], Y8[8];
  codes_from_planes<Q>(pw_, Yg, Y8);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int d = rt * 16 + g + 8 * r;
    const int row = orig_row(d, u, I);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = kc * 128 + 16 * s + 2 * c + (e & 1) + 8 * (e >> 1);
        if (col >= bd.K) continue;
        const uint32_t code = code_at<Q>(r ? Y8[s] : Yg[s], e);
        if (idx_out) idx_out[(size_t)row * bd.K + col] = (uint8_t)code;
        if (w_out) w_out[(size_t)row * bd.K + col] = bd.lut[Q][(size_t)d * (1 << Q) + code];
      }
    }
  }
}

__global__ void unpack_kernel(const BlockDev *table, int block, int b, int u, int I,
                              uint8_t *idx_out, uint16_t *w_out) {
  const BlockDev &bd = table[block];
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int ntk = (bd.N / 16) * bd.KC;
  if (warp_global >= ntk) return;
  const int rt = warp_global / bd.KC, kc = warp_global % bd.KC;
  switch (b) {
    case 1: unpack_chunk<1>(bd, rt, kc, u, I, idx_out, w_out); break;
    case 2: unpack_chunk<2>(bd, rt, kc, u, I, idx_out, w_out); break;
    case 3: unpack_chunk<3>(bd, rt, kc, u, I, idx_out, w_out); break;
    case 4: unpack_chunk<4>(bd, rt, kc, u, I, idx_out, w_out); break;
    case 5: unpack_chunk<5>(bd, rt, kc, u, I, idx_out, w_out); break;
    case 6: unpack_chunk<6>(bd, rt, kc, u, I, idx_out, w_out); break;
    case 7: unpack_chunk<7>(bd, rt, kc, u, I, idx_out, w_out); break;
    default: unpack_chunk<8>(bd, rt, kc, u, I, idx_out, w_out); break;
  }
}

int launch_unpack(const BlockDev *table, int block, int b, int u, int I, int N, int KC,
                        uint8_t *idx_out, uint16_t *w_out, void *stream) {
  const long warps = (long)(N / 16) * KC;
  const int thr = 128;
  const long blocks = (warps * 32 + thr - 1) / thr;
  unpack_kernel<<<(unsigned)blocks, thr, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      table, block, b, u, I, idx_out, w_out);
  return (int)cudaGetLastError();
}

int launch_fill_u32(uint32_t *p, uint32_t v, long n, void *stream) {
  return (int)cudaMemsetAsync(p, (int)(v & 0xFF), (size_t)n * 4, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace pw

namespace pw {
// The router kernel alone (logits, softmax, top-K, bucketing) on scratch the caller chose.
int launch_route(const FwdArgs &a, void *stream_) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtTok * 8192 * 2);
  dim3 rg((a.T + kRtTok - 1) / kRtTok, (a.E + kRtExp - 1) / kRtExp);
  route_kernel<<<rg, kRtThreads, kRtTok * a.H * 2, st>>>(a);
  return (int)cudaGetLastError();
}
}  // namespace pw
