// pw_kernels.cu -- combine and bookkeeping kernels of the fused mixed-precision MoE
// layer (sm_103a); the router is in pw_route.cu, the expert kernels in pw_ffn.cu.
//
// PagedWeight Sec. 3.3 ("Fused Mixed-Precision MoE Kernel"): routing, expert activation,
// down projection and output accumulation, each linear block read directly from its AP
// bit-planes and LUT at its committed bitwidth.  One layer is four launches:
//   route_kernel   router logits (fp32), softmax, top-K; writes the experts' fp16 input;
//                  the last CTA to finish buckets the (token, k) pairs by expert and writes
//                  the work lists and routing statistics
//   ffn (phase 1)  gate_up of every active expert and of the shared expert, SiLU(g)*u
//   ffn (phase 2)  down projection of every active expert and of the shared expert
//   combine_kernel y_t = sum_k r_tk o_tk (k order; o_tk the sum of its K parts in order)
//                  + shared (+ y when accumulating)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw_device.cuh"
#include "pw_dq.cuh"
#include "pw_internal.h"

namespace pw {

// ------------------------------------------------------------------ combine
__global__ void __launch_bounds__(256) combine_kernel(FwdArgs a) {
  pdl_trigger();
  pdl_wait();
  // both expert kernels of the layer have completed: their claim counters and the layer's
  // ready counts start over (the next expert kernel claims only after the next router has
  // counted its rows, and that router waits for this kernel)
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    a.s.work[0] = 0;
    a.s.work[1] = 0;
    if (a.s.ready) {
      a.s.ready[2 * a.layer] = 0;
      a.s.ready[2 * a.layer + 1] = 0;
    }
  }
  const int t = blockIdx.x;
  const int h_begin = blockIdx.y * 1024, h_end = min(a.H, h_begin + 1024);
  const int H = a.H, K = a.K;
  __shared__ int s_slot[8];
  __shared__ float s_w[8];
  if (threadIdx.x < K) {
    s_slot[threadIdx.x] = a.s.pair_slot[t * K + threadIdx.x];
    s_w[threadIdx.x] = a.s.w[t * K + threadIdx.x];
  }
  __syncthreads();
  const int np = routed_down_splits(a.T, a.I);  // K parts of the routed down projection
  const size_t pstride = (size_t)a.T * K * H;
  for (int h = h_begin + threadIdx.x * 4; h < h_end; h += 256 * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (np == 1) {
      for (int k = 0; k < K; ++k) {
        const float4 o = *reinterpret_cast<const float4 *>(a.s.o_routed + (size_t)s_slot[k] * H + h);
        const float r = s_w[k];
        acc.x = fmaf(r, o.x, acc.x);
        acc.y = fmaf(r, o.y, acc.y);
        acc.z = fmaf(r, o.z, acc.z);
        acc.w = fmaf(r, o.w, acc.w);
      }
    } else {
      for (int k = 0; k < K; ++k) {
        const float *op = a.s.o_routed + (size_t)s_slot[k] * H + h;
        float4 o = *reinterpret_cast<const float4 *>(op);
        for (int p = 1; p < np; ++p) {  // the parts' partial sums, in order
          const float4 ov = *reinterpret_cast<const float4 *>(op + p * pstride);
          o.x += ov.x;
          o.y += ov.y;
          o.z += ov.z;
          o.w += ov.w;
        }
        const float r = s_w[k];
        acc.x = fmaf(r, o.x, acc.x);
        acc.y = fmaf(r, o.y, acc.y);
        acc.z = fmaf(r, o.z, acc.z);
        acc.w = fmaf(r, o.w, acc.w);
      }
    }
    if (a.Is > 0) {  // the shared expert's partial sums, in order
      const int nsplit = shared_down_splits(a.I, a.Is);
      float4 sh = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p = 0; p < nsplit; ++p) {
        const float4 sv = *reinterpret_cast<const float4 *>(a.s.o_shared + ((size_t)p * a.T + t) * H + h);
        sh.x += sv.x;
        sh.y += sv.y;
        sh.z += sv.z;
        sh.w += sv.w;
      }
      const float g = a.lay.wsg ? a.s.sgate[t] : 1.f;  // the shared-expert gate, when the layer has one
      acc.x = fmaf(g, sh.x, acc.x);
      acc.y = fmaf(g, sh.y, acc.y);
      acc.z = fmaf(g, sh.z, acc.z);
      acc.w = fmaf(g, sh.w, acc.w);
    }
    uint2 *yp = reinterpret_cast<uint2 *>(a.y + (size_t)t * H + h);
    if (a.flags & 1) {
      const uint2 old = *yp;
      acc.x += bf16f(old.x & 0xFFFF);
      acc.y += bf16f(old.x >> 16);
      acc.z += bf16f(old.y & 0xFFFF);
      acc.w += bf16f(old.y >> 16);
    }
    const uint2 yv = make_uint2(pack2(f2bf(acc.x), f2bf(acc.y)), pack2(f2bf(acc.z), f2bf(acc.w)));
    *yp = yv;
    // a bf16 whose exponent bits are all ones is an infinity or a NaN
    const bool fin = (~yv.x & 0x7F80u) && (~yv.x & 0x7F800000u) && (~yv.y & 0x7F80u) && (~yv.y & 0x7F800000u);
    if (!fin) atomicOr(a.s.err, kErrRange);
  }
}

__device__ __forceinline__ void store_item(WorkItem *dst, const WorkItem &w) {
  int4 *p = reinterpret_cast<int4 *>(dst);
  p[0] = make_int4(w.kind, w.expert, w.tile, w.tok0);
  p[1] = make_int4(w.ntok, w.kc0, w.kc1, w.part);
}

// The layer's routing statistics, added to the running sums of row a.stat_layer: per expert
// the number of its (token, k) selections and the sum of their routing weights r (Eq. 1's
// inputs), and the sums behind Eq. 5's routed-input features (sum r n, sum r n^2, max n; n =
// the slot token's input norm as the experts read it).  G lanes per expert stride over its
// slots [offsets[e], offsets[e + 1]) and a shuffle tree adds their sums, so the order is
// fixed.  An expert holds at most T slots: decode batches take G = 4, larger ones a warp.
template <int G>
__device__ void routing_statistics(const FwdArgs &a) {
  const int E = a.E, lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int sub = lane / G, gl = lane % G;
  for (int eb = warp * (32 / G); eb < E; eb += nw * (32 / G)) {
    const int e = eb + sub;
    const size_t si = (size_t)a.stat_layer * E + (e < E ? e : 0);
    // the running sums and the slot range load together
    double st_c = 0., st_w = 0., st_p[4] = {0., 0., 0., 0.};
    int o0 = 0, o1 = 0;
    if (e < E && gl == 0) {
      st_c = a.s.stat_count[si];
      st_w = a.s.stat_wsum[si];
      if (a.s.stat_phi)
#pragma unroll
        for (int i = 0; i < 4; ++i) st_p[i] = a.s.stat_phi[si * 4 + i];
    }
    if (e < E) {
      o0 = a.s.offsets[e];
      o1 = a.s.offsets[e + 1];
    }
    float wsum = 0.f, s1 = 0.f, s2 = 0.f, mx = 0.f;
#pragma unroll 4
    for (int sl = o0 + gl; sl < o1; sl += G) {
      const float r = a.s.slot_w[sl];
      const float n = a.s.xnorm[a.s.slot_tok[sl]];
      wsum += r;
      s1 = fmaf(r, n, s1);
      s2 = fmaf(r * n, n, s2);
      mx = fmaxf(mx, n);
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
      wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (e < E && gl == 0) {
      const int cnt = o1 - o0;
      a.s.stat_count[si] = st_c + (double)cnt;
      a.s.stat_wsum[si] = st_w + (double)wsum;
      if (a.s.stat_phi && cnt > 0) {
        double *ph = a.s.stat_phi + si * 4;
        ph[0] = st_p[0] + (double)wsum;
        ph[1] = st_p[1] + (double)s1;
        ph[2] = st_p[2] + (double)s2;
        ph[3] = fmax(st_p[3], (double)mx);
      }
    }
  }
}

// Three jobs between the router and the expert kernels, grid-stride over every CTA:
//  * the layer input's rows in expert-sorted slot order (xs[slot] = xh[token of slot]), so
//    that every routed gate_up work item reads consecutive rows with TMA boxes (16-byte
//    vectors);
//  * the work items of both projections, expanded from the router's work-list tables (one
//    thread per item);
//  * in the last CTA, the layer's routing statistics.
// The tables' loads are issued first and land while the rows are copied.
__global__ void __launch_bounds__(256) gather_kernel(FwdArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ int s_first[2][kRankStride], s_rk[2][kRankStride], s_off[kRankStride];
  const int E = a.E, tid = threadIdx.x;  // blockDim.x == 256 >= E
  const int *R = a.s.ranks;
  int f0 = 0, f1 = 0, k0 = 0, k1 = 0, of = 0, fE0 = 0, fE1 = 0, oE = 0;
  if (tid <= E) {
    f0 = R[tid];
    f1 = R[kRankStride + tid];
    of = a.s.offsets[tid];
  }
  if (tid < E) {
    k0 = R[2 * kRankStride + tid];
    k1 = R[3 * kRankStride + tid];
  }
  const bool last = tid == 0 && E == 256;  // entry E of first and offsets when E == blockDim.x
  if (last) {
    fE0 = R[E];
    fE1 = R[kRankStride + E];
    oE = a.s.offsets[E];
  }
  const int vec = a.H / 8;
  const long n = (long)a.T * a.K * vec;
  for (long i = (long)blockIdx.x * blockDim.x + tid; i < n; i += (long)gridDim.x * blockDim.x) {
    const int s = (int)(i / vec), v = (int)(i % vec);
    const int t = a.s.slot_tok[s];
    reinterpret_cast<uint4 *>(a.s.xs + (size_t)s * a.H)[v] = reinterpret_cast<const uint4 *>(a.s.xh + (size_t)t * a.H)[v];
  }
  if (tid <= E) {
    s_first[0][tid] = f0;
    s_first[1][tid] = f1;
    s_off[tid] = of;
  }
  if (tid < E) {
    s_rk[0][tid] = k0;
    s_rk[1][tid] = k1;
  }
  if (last) {
    s_first[0][E] = fE0;
    s_first[1][E] = fE1;
    s_off[E] = oE;
  }
  __syncthreads();
  const int n1 = s_first[0][E], n_all = n1 + s_first[1][E];
  for (int i = blockIdx.x * blockDim.x + tid; i < n_all; i += gridDim.x * blockDim.x) {
    const int u = i >= n1 ? 1 : 0, iu = u ? i - n1 : i;
    store_item((u ? a.s.items2 : a.s.items1) + iu,
               work_item(u, iu, s_first[u], s_rk[u], s_off, E, a.T, a.H, a.I, a.Is));
  }
  if (blockIdx.x == gridDim.x - 1) {
    if (a.T <= 256)
      routing_statistics<4>(a);
    else
      routing_statistics<32>(a);
  }
}

// ------------------------------------------------------------------ launch
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
  if (ev) record(ev[0], st);
  if (int e = launch_route(a, stream_)) return e;
  if (!a.s.xs) return (int)cudaErrorInvalidValue;
  {
    const long vecs = (long)a.T * a.K * (a.H / 8);
    const long want = (vecs + 255) / 256, cap = (long)a.sm_count * 4;
    const int blocks = (int)(want < cap ? want : cap);
    if (cudaError_t e = launch_pdl(gather_kernel, dim3(blocks), dim3(256), 0, st, a)) return (int)e;
  }
  if (ev) record(ev[1], st);
  if (int e = launch_ffn(a, 1, stream_)) return e;
  if (ev) record(ev[2], st);
  if (int e = launch_ffn(a, 2, stream_)) return e;
  if (ev) record(ev[3], st);
  if (cudaError_t e = launch_pdl(combine_kernel, dim3(a.T, (a.H + 1023) / 1024), dim3(256), 0, st, a)) return (int)e;
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

// One thread per (CTA tile, chunk, column group, row); writes that word of every plane.
__global__ void pack_kernel(const uint8_t *idx, int N, int K, int KC, int u, int I, int bmax,
                            uint32_t *const *planes, long nwords) {
  const long li = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (li >= nwords) return;
  const long full = (long)kCtaRows * KC * 4;  // words of a full CTA tile
  const int ct = (int)(li / full);
  const int nr = tile_rows(ct, N);
  const int off = (int)(li - ct * full);
  const int kc = off / (nr * 4), rem = off % (nr * 4);
  const int cg = rem / nr, r = rem % nr;
  const int row = orig_row(ct * kCtaRows + r, u, I);
  uint32_t words[kMaxPlanes] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int b = 0; b < 32; ++b) {
    const int col = kc * kChunkCols + 32 * cg + 8 * (b & 3) + (b >> 2);
    const uint32_t code = (col < K) ? idx[(size_t)row * K + col] : 0u;
    for (int p = 0; p < bmax; ++p) words[p] |= ((code >> (bmax - 1 - p)) & 1u) << b;
  }
  for (int p = 0; p < bmax; ++p) planes[p][li] = words[p];
}

int launch_pack(const uint8_t *idx, int N, int K, int KC, int u, int I, int bmax,
                uint32_t *const *plane_out, void *stream) {
  const long nwords = (long)N * KC * 4;  // 4 words (128 bits) per row and chunk
  const int thr = 256;
  const long blocks = (nwords + thr - 1) / thr;
  pack_kernel<<<(unsigned)blocks, thr, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      idx, N, K, KC, u, I, bmax, plane_out, nwords);
  return (int)cudaGetLastError();
}

// LUT_b from the caller's [N][2^b] (original rows) to the kernel-private tiled layout
// (lut_dev_index; rows of the padded last tile are zero).  One thread per output entry.
__global__ void lut_permute_kernel(const uint16_t *in, int N, int b, int u, int I, uint16_t *out, long total) {
  const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const long tile = lut_tile_bytes(b) / 2;
  const int ct = (int)(i / tile);
  const long rem = i % tile;
  const int half = (int)(rem & 1);
  const long word = rem >> 1;
  const int c = (int)(word / 64), w64 = (int)(word % 64);
  const int m = 2 * (w64 / 32) + half, L = w64 % 32;
  const int d = ct * kCtaRows + 32 * m + L;
  out[i] = d < N ? in[(size_t)orig_row(d, u, I) * (1 << b) + c] : (uint16_t)0;
}

int launch_lut_permute(const uint16_t *lut_in, int N, int entries, int u, int I, uint16_t *lut_out,
                       void *stream) {
  int b = 0;
  while ((1 << b) < entries) ++b;
  const long n = lut_dev_bytes(N, b) / 2;
  lut_permute_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      lut_in, N, b, u, I, lut_out, n);
  return (int)cudaGetLastError();
}

// bf16 -> fp16 in the shared-weight operand-tile layout (the output is pre-zeroed, so the
// padding rows and columns stay zero); counts values that overflow fp16 into *bad.
__global__ void frag16_kernel(const uint16_t *in, int N, int K, int u, int I, uint16_t *out, int *bad) {
  long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long)N * K) return;
  const int d = (int)(i / K), k = (int)(i % K);
  const float v = bf16f(in[(size_t)orig_row(d, u, I) * K + k]);
  if (!(fabsf(v) <= 65504.0f)) atomicAdd(bad, 1);
  out[shared_tile_index(d, k, K)] = f2h(v);
}

int launch_frag16(const uint16_t *w_in, int N, int K, int u, int I, uint16_t *w_out, int *bad, void *stream) {
  const long n = (long)N * K;
  frag16_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      w_in, N, K, u, I, w_out, bad);
  return (int)cudaGetLastError();
}

// Debug read-back through the forward's dequantisation code (pw_dq.cuh): one CTA per
// (CTA tile, chunk), one thread per (column group, row); the tile's LUT is staged in shared
// memory at a 64 KB-aligned address as in the expert kernels.
template <int Q>
__device__ void unpack_group(const BlockDev &bd, int ct, int kc, int cg, int r, int u, int I, uint32_t lut_s,
                             uint8_t *idx_out, uint16_t *w_out) {
  const int nr = tile_rows(ct, bd.N);
  const long w0 = slab_word(ct, kc, bd.N, bd.KC) + (long)cg * nr + r;
  uint32_t W[8];
#pragma unroll
  for (int p = 0; p < 8; ++p) W[p] = p < Q ? bd.plane[p][w0] : 0u;
  const int d = ct * kCtaRows + r;
  const LutLane lu = lut_lane(lut_s, r / 32, r % 32);
  uint32_t v[16], codes[32];
  if constexpr (Q <= kRegLutMaxQ) {
    uint32_t S[4], P[8];
    codes_nib<Q>(W, S);
    lut_pairs_smem<Q>(lu, P);
    LutRegs L;
    lut_regs(P, L);
    dq_nib<Q>(S, L, v);
#pragma unroll
    for (int c = 0; c < 32; ++c) codes[c] = code_nib<Q>(S, c);
  } else {
    uint32_t Y[8];
    codes_byte<Q>(W, Y, lu.top);
    dq_byte<Q>(Y, lu, v);
#pragma unroll
    for (int c = 0; c < 32; ++c) codes[c] = code_byte<Q>(Y, c);
  }
  const int row = orig_row(d, u, I);
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const int col = kc * kChunkCols + 32 * cg + c;
    if (col >= bd.K) continue;
    if (idx_out) idx_out[(size_t)row * bd.K + col] = (uint8_t)codes[c];
    if (w_out) w_out[(size_t)row * bd.K + col] = (uint16_t)((c & 1) ? (v[c >> 1] >> 16) : (v[c >> 1] & 0xFFFFu));
  }
}

constexpr int kUnpackSmem = 128 * 1024;  // a 64 KB-aligned 64 KB window inside

__global__ void __launch_bounds__(512) unpack_kernel(const BlockDev *table, int block, int b, int u, int I,
                                                     uint8_t *idx_out, uint16_t *w_out) {
  extern __shared__ __align__(1024) uint8_t lut_smem[];
  const BlockDev &bd = table[block];
  const int ct = blockIdx.x, kc = blockIdx.y;
  const int nr = tile_rows(ct, bd.N);
  const int cg = threadIdx.x / kCtaRows, r = threadIdx.x % kCtaRows;
  const uint32_t lut_s = (smem_u32(lut_smem) + 65535u) & ~65535u;
  {  // stage the tile's LUT as the expert kernels do
    const int n16 = (int)(lut_tile_bytes(b) / 16);
    const uint4 *src = reinterpret_cast<const uint4 *>(bd.lut[b] + ct * (lut_tile_bytes(b) / 2));
    uint4 *dst = reinterpret_cast<uint4 *>(lut_smem + (lut_s - smem_u32(lut_smem)));
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = src[i];
  }
  __syncthreads();
  if (r >= nr) return;
  switch (b) {
    case 1: unpack_group<1>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
    case 2: unpack_group<2>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
    case 3: unpack_group<3>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
    case 4: unpack_group<4>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
    case 5: unpack_group<5>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
    case 6: unpack_group<6>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
    case 7: unpack_group<7>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
    default: unpack_group<8>(bd, ct, kc, cg, r, u, I, lut_s, idx_out, w_out); break;
  }
}

int launch_unpack(const BlockDev *table, int block, int b, int u, int I, int N, int KC, uint8_t *idx_out,
                  uint16_t *w_out, void *stream) {
  cudaFuncSetAttribute(unpack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUnpackSmem);
  dim3 grid((N + kCtaRows - 1) / kCtaRows, KC);
  unpack_kernel<<<grid, 4 * kCtaRows, kUnpackSmem, reinterpret_cast<cudaStream_t>(stream)>>>(table, block, b, u, I,
                                                                                             idx_out, w_out);
  return (int)cudaGetLastError();
}

}  // namespace pw
