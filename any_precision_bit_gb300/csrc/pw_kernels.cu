// pw_kernels.cu -- router, combine and bookkeeping kernels of the fused mixed-precision MoE
// layer (sm_103a); the expert kernels are in pw_ffn.cu.
//
// PagedWeight Sec. 3.3 ("Fused Mixed-Precision MoE Kernel"): routing, expert activation,
// down projection and output accumulation, each linear block read directly from its AP
// bit-planes and LUT at its committed bitwidth.  One layer is four launches:
//   route_kernel   router logits (fp32), softmax, top-K; writes the experts' fp16 input;
//                  the last CTA to finish buckets the (token, k) pairs by expert and writes
//                  the work lists and routing statistics
//   ffn (phase 1)  gate_up of every active expert and of the shared expert, SiLU(g)*u
//   ffn (phase 2)  down projection of every active expert and of the shared expert
//   combine_kernel y_t = sum_k r_tk o_tk (k order) + shared (+ y when accumulating)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw_device.cuh"
#include "pw_internal.h"

namespace pw {

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
  if (blockIdx.y == 0) {  // the experts' fp16 input rows
    for (int v = tid; v < nt * H / 8; v += kRtThreads) {
      const int t = v / (H / 8), c = (v % (H / 8)) * 8;
      const uint4 raw = *reinterpret_cast<const uint4 *>(xs + t * H + c);
      const float inv = s_inv[t];
      const uint32_t r[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = pack2(f2h(bf16f(r[i]) * inv), f2h(bf16f(r[i] >> 16) * inv));
      *reinterpret_cast<uint4 *>(a.s.xh + (size_t)(t0 + t) * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  const int e = blockIdx.y * kRtExp + warp;
  if (e < E) {
    float acc[kRtTok];
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) acc[t] = 0.f;
    const float *wr = a.lay.Wr + (size_t)e * H;
    // issue the whole router row's loads before using any (H <= 8192: <= 16 per lane, 4 at a time)
#pragma unroll 4
    for (int h = lane * 4; h < H; h += 128) {
      float4 wv = __ldg(reinterpret_cast<const float4 *>(wr + h));
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
  // the logits (written by other CTAs, so read through L2), staged in shared memory when they
  // fit: every load is then in flight at once instead of one round trip per token
  const bool staged = (size_t)T * E * 4 <= (size_t)kRtTok * H * 2;
  float *sl = reinterpret_cast<float *>(smem_raw);
  if (staged) {
    for (int i = tid; i < T * E; i += kRtThreads) sl[i] = __ldcg(a.s.logits + i);
    __syncthreads();
  }
  // softmax + top-K, one warp per token
  for (int t = warp; t < T; t += kRtThreads / 32) {
    const float *lg = staged ? sl + (size_t)t * E : a.s.logits + (size_t)t * E;
    float lv[8];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int ee = lane + 32 * i;
      lv[i] = (ee < E) ? (staged ? lg[ee] : __ldcg(lg + ee)) : -INFINITY;
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
  const int nsplit = shared_down_splits(a.I, a.Is);
  const int sh1 = a.Is > 0 ? ((2 * a.Is + kCtaRows - 1) / kCtaRows) * tchunks : 0;
  const int sh2 = a.Is > 0 ? tiles2 * tchunks * nsplit : 0;
  const int kc_gu = kpad_cols(a.H) / kChunkCols, kc_d = kpad_cols(a.I) / kChunkCols;
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
    a.s.items1[i] = WorkItem{1, 0, tile, ch * kTokChunk, min(kTokChunk, T - ch * kTokChunk),
                             0, (a.H / 16 + 7) / 8, 0};
  }
  {
    const int total = (a.Is / 16 + 7) / 8, per = (total + nsplit - 1) / nsplit;
    for (int i = tid; i < sh2; i += kRtThreads) {
      const int tile = i / (tchunks * nsplit), rem = i % (tchunks * nsplit);
      const int ch = rem / nsplit, part = rem % nsplit;
      a.s.items2[i] = WorkItem{1, 0, tile, ch * kTokChunk, min(kTokChunk, T - ch * kTokChunk),
                               part * per, min(total, (part + 1) * per), part};
    }
  }
  __syncthreads();
  // routed work items and routing statistics, one thread per expert
  for (int ee = tid; ee < E; ee += kRtThreads) {
    const int cnt = s_cnt[ee];
    const int ch = (cnt + kTokChunk - 1) / kTokChunk;
    int p1 = s_itm1[ee], p2 = s_itm2[ee];
    for (int c = 0; c < ch; ++c) {
      int nt2 = min(kTokChunk, cnt - c * kTokChunk);
      for (int tile = 0; tile < tiles1; ++tile)
        a.s.items1[p1++] = WorkItem{0, ee, tile, c * kTokChunk, nt2, 0, kc_gu, 0};
      for (int tile = 0; tile < tiles2; ++tile)
        a.s.items2[p2++] = WorkItem{0, ee, tile, c * kTokChunk, nt2, 0, kc_d, 0};
    }
  }
  __syncthreads();
  // routing statistics: one warp per expert, the expert's slots summed in a fixed order
  for (int ee = warp; ee < E; ee += kRtThreads / 32) {
    const int cnt = s_cnt[ee], o0 = s_off[ee];
    double ws = 0.0;
    for (int sl = lane; sl < cnt; sl += 32) ws += (double)a.s.slot_w[o0 + sl];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    if (lane == 0) {
      a.s.stat_count[(size_t)a.layer * E + ee] += (double)cnt;
      a.s.stat_wsum[(size_t)a.layer * E + ee] += ws;
    }
  }
  if (tid == 0) *a.s.ticket = 0u;
}

// ------------------------------------------------------------------ combine
__global__ void __launch_bounds__(256) combine_kernel(FwdArgs a) {
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
  for (int h = h_begin + threadIdx.x * 4; h < h_end; h += 256 * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      const float4 o = *reinterpret_cast<const float4 *>(a.s.o_routed + (size_t)s_slot[k] * H + h);
      const float r = s_w[k];
      acc.x = fmaf(r, o.x, acc.x);
      acc.y = fmaf(r, o.y, acc.y);
      acc.z = fmaf(r, o.z, acc.z);
      acc.w = fmaf(r, o.w, acc.w);
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
      acc.x += sh.x;
      acc.y += sh.y;
      acc.z += sh.z;
      acc.w += sh.w;
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

int launch_route(const FwdArgs &a, void *stream_) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtTok * 8192 * 2);
  dim3 rg((a.T + kRtTok - 1) / kRtTok, (a.E + kRtExp - 1) / kRtExp);
  route_kernel<<<rg, kRtThreads, kRtTok * a.H * 2, st>>>(a);
  return (int)cudaGetLastError();
}

int launch_forward(const FwdArgs &a, void *stream_, void *const *ev_) {
  cudaEvent_t const *ev = reinterpret_cast<cudaEvent_t const *>(ev_);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  if (ev) record(ev[0], st);
  if (int e = launch_route(a, stream_)) return e;
  if (ev) record(ev[1], st);
  if (int e = launch_ffn(a, 1, stream_)) return e;
  if (ev) record(ev[2], st);
  if (int e = launch_ffn(a, 2, stream_)) return e;
  if (ev) record(ev[3], st);
  combine_kernel<<<dim3(a.T, (a.H + 1023) / 1024), 256, 0, st>>>(a);
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

// One thread per (warp tile, chunk, lane, row half); writes that word of every plane.
__global__ void pack_kernel(const uint8_t *idx, int N, int K, int KC, int u, int I, int bmax,
                            uint32_t *const *planes, long nwords) {
  long li = (long)blockIdx.x * blockDim.x + threadIdx.x;
  if (li >= nwords) return;
  const int r = (int)(li & 1);
  const int lane = (int)((li >> 1) & 31);
  const long tk = li >> 6;
  const int kc = (int)(tk % KC);
  const int rt = (int)(tk / KC);
  const int d = rt * 16 + 8 * r + (lane & 7);
  const int row = orig_row(d, u, I);
  uint32_t words[kMaxPlanes] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int e = 0; e < 4; ++e) {
    for (int s = 0; s < 8; ++s) {
      const int col = kc * 128 + 32 * (lane >> 3) + 4 * s + e;
      const uint32_t code = (col < K) ? idx[(size_t)row * K + col] : 0u;
      for (int p = 0; p < bmax; ++p) words[p] |= ((code >> (bmax - 1 - p)) & 1u) << (8 * e + s);
    }
  }
  const long dst = plane_pair_word(rt, kc, N / 16, KC) + lane * 2 + r;
  for (int p = 0; p < bmax; ++p) planes[p][dst] = words[p];
}

int launch_pack(const uint8_t *idx, int N, int K, int KC, int u, int I, int bmax,
                uint32_t *const *plane_out, void *stream) {
  const long nwords = (long)N * KC * 4;  // N/16 warp tiles * KC chunks * 64 words
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

// Debug read-back through the forward's extraction code: one warp per (warp tile, chunk).
template <int Q>
__device__ void unpack_chunk(const BlockDev &bd, int rt, int kc, int u, int I, uint8_t *idx_out,
                             uint16_t *w_out) {
  const int lane = threadIdx.x & 31;
  const long base = plane_pair_word(rt, kc, bd.N / 16, bd.KC) / 2 + lane;
  uint2 pw_[Q];
#pragma unroll
  for (int p = 0; p < Q; ++p) pw_[p] = reinterpret_cast<const uint2 *>(bd.plane[p])[base];
  uint32_t Yg[8], Y8[8];
  codes_from_planes<Q>(pw_, Yg, Y8);
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int d = rt * 16 + 8 * r + (lane & 7);
    const int row = orig_row(d, u, I);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = kc * 128 + 32 * (lane >> 3) + 4 * s + e;
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

int launch_unpack(const BlockDev *table, int block, int b, int u, int I, int N, int KC, uint8_t *idx_out,
                  uint16_t *w_out, void *stream) {
  const long warps = (long)(N / 16) * KC;
  const int thr = 128;
  const long blocks = (warps * 32 + thr - 1) / thr;
  unpack_kernel<<<(unsigned)blocks, thr, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      table, block, b, u, I, idx_out, w_out);
  return (int)cudaGetLastError();
}

}  // namespace pw
