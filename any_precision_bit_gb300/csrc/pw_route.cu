// pw_route.cu -- the router of the fused mixed-precision MoE layer (sm_103a).
//
// PagedWeight Sec. 3.3 ("Fused Mixed-Precision MoE Kernel"): routing is the first step of
// the fused layer.  One launch, grid (token groups of kRtTok) x (expert groups of kRtExp):
//   every CTA        bulk-copies its kRtTok token rows and kRtExp router rows into shared
//                    memory, takes the tokens' 1/rms (PW_PRENORM), writes its column slice of
//                    the experts' fp16 input rows and the fp32 logits of its experts (the
//                    last expert group also the shared expert's gate);
//   last CTA of a    (elected by a per-group atomic ticket once every expert group wrote its
//   token group      logits) takes softmax and top-K of the group's tokens, one warp each;
//   last CTA of all  (elected by a second ticket once every token group is ranked) buckets
//                    the (token, k) pairs by expert in the stable (expert, token, k) order
//                    and writes the tables of the expert kernels' work lists.
// The single-CTA tail is short by construction: top-K runs in as many CTAs as there are
// token groups, the bucket ranks come from warp-private match_any counts and block scans,
// the work items are expanded from the tables by the many CTAs of the gather kernel, which
// also adds the layer's routing statistics (the inputs of Eq. 1 and Eq. 5) off this path,
// and the tail's global loads (pairs, bitwidths) are issued in batches so that their
// latencies overlap instead of adding up.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw_device.cuh"
#include "pw_internal.h"

namespace pw {

constexpr int kRtThreads = 256;
constexpr int kRtWarps = kRtThreads / 32;
constexpr int kRtStageBytes = 96 * 1024;  // token rows + one column chunk of the router rows
constexpr int kRtMaxSmem = 160 * 1024;
constexpr long kRtSpin = 1L << 22;

// Columns of the router rows staged at once: the token rows (kRtTok x H bf16) stay whole,
// the router rows (kRtExp x Hc fp32) go in chunks of Hc columns.
__host__ __device__ inline int route_hchunk(int H) {
  int hc = (kRtStageBytes - kRtTok * H * 2) / (kRtExp * 4);
  hc = hc / 128 * 128;
  if (hc < 512) hc = 512;
  return hc < H ? hc : H;
}

// Dynamic shared memory of a router launch: the staged rows, or the pair arrays [ids][weights]
// that the last CTA keeps there when they fit in kRtStageBytes (or in the stage, if larger).
struct RouteSmem {
  int bytes;
  bool pairs;
};
__host__ __device__ inline RouteSmem route_smem(int T, int K, int H) {
  RouteSmem r;
  const int stage = kRtTok * H * 2 + kRtExp * route_hchunk(H) * 4;
  const int cap = stage > kRtStageBytes ? stage : kRtStageBytes;
  const int pair_bytes = T * K * 8;
  r.pairs = pair_bytes <= cap;
  r.bytes = r.pairs && pair_bytes > stage ? pair_bytes : stage;
  return r;
}

// Ranking key of expert e with logit l: a larger key ranks higher, NaN ranks below every
// number (-inf included) and equal logits rank the lower id first.  Keys of distinct
// experts differ and no key is 0.  Softmax is increasing, so ranking logits ranks the
// routing probabilities.
__device__ __forceinline__ uint64_t rank_key(float l, int e) {
  uint32_t b = __float_as_uint(l);
  if (l == 0.f) b = 0u;  // -0 and +0 are the same logit
  const uint32_t ord = (l != l) ? 0u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
  return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
}
__device__ __forceinline__ float key_logit(uint64_t key) {
  const uint32_t ord = (uint32_t)(key >> 32);
  return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}
__device__ __forceinline__ int key_expert(uint64_t key) { return (int)(0xFFFFFFFFu - (uint32_t)key); }

// keep the 8 largest keys seen, in descending order
__device__ __forceinline__ void top8_insert(uint64_t (&v)[8], uint64_t key) {
  if (key <= v[7]) return;
  v[7] = key;
#pragma unroll
  for (int s = 7; s > 0; --s)
    if (v[s] > v[s - 1]) {
      const uint64_t t = v[s];
      v[s] = v[s - 1];
      v[s - 1] = t;
    }
}

// Softmax and top-K of token t, one warp: each lane takes experts lane, lane + 32, ... with
// a running max and a top-8 list; the lists merge over the warp one rank at a time.
__device__ void softmax_topk_warp(const FwdArgs &a, int t, int lane) {
  const int E = a.E, K = a.K;
  const float *lg = a.s.logits + (size_t)t * E;
  uint64_t v[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) v[s] = 0ull;
  float m = -INFINITY, s = 0.f;  // running max and sum of exp(l - m) over this lane's experts
  float lv[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {  // E <= 256: at most 8 experts per lane, all loads in flight
    const int ee = lane + 32 * u;
    lv[u] = ee < E ? __ldcg(lg + ee) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int ee = lane + 32 * u;
    if (ee < E) {
      const float l = lv[u];
      top8_insert(v, rank_key(l, ee));
      if (l > m) {
        s = s * expf(m - l) + 1.f;
        m = l;
      } else if (l != -INFINITY) {  // exp(-inf) adds nothing; NaN propagates
        s += expf(l - m);
      }
    }
  }
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float S = (s == 0.f) ? 0.f : s * expf(m - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
  const float inv = 1.0f / S;
  float pk = 0.f, csum = 0.f;  // lane k keeps rank k
  int ik = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k < K) {
      uint64_t best = v[0];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const uint64_t ob = __shfl_xor_sync(0xffffffffu, best, o);
        best = ob > best ? ob : best;
      }
      if (best != 0ull && v[0] == best) {  // the lane holding the winner drops it
#pragma unroll
        for (int q = 0; q < 7; ++q) v[q] = v[q + 1];
        v[7] = 0ull;
      }
      const float p = expf(key_logit(best) - M) * inv;
      csum += p;
      if (lane == k) {
        pk = p;
        ik = best != 0ull ? min(key_expert(best), E - 1) : E - 1;
      }
    }
  }
  if (lane < K) {
    const float wv = a.renorm ? pk / csum : pk;
    const int j = t * K + lane;
    a.s.ids[j] = ik;
    a.s.w[j] = wv;
    if (a.ids_out) a.ids_out[j] = ik;
    if (a.w_out) a.w_out[j] = wv;
  }
}

// Two CTAs per SM at most (the staged rows take up to 96 KB of shared memory each), so the
// register budget is half the register file per CTA.
__global__ void __launch_bounds__(kRtThreads, 2) route_kernel(FwdArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int H = a.H, E = a.E, K = a.K;
  const int hc = route_hchunk(H);
  uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);                 // [kRtTok][H] bf16
  float *ws = reinterpret_cast<float *>(smem_raw + kRtTok * H * 2);      // [kRtExp][hc] fp32
  __shared__ __align__(8) uint64_t bar;
  __shared__ float s_inv[kRtTok];
  __shared__ int s_flag;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * kRtTok, nt = min(kRtTok, a.T - t0);
  const int e0 = blockIdx.y * kRtExp, ne = min(kRtExp, E - e0);
  const uint32_t b = smem_u32(&bar);
  if (tid == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // the previous kernel of the stream (the last layer's combine) wrote x and still reads the
  // routing scratch this kernel rewrites
  pdl_trigger();
  pdl_wait();

  // ---- logits: token rows once, router rows chunk by chunk (bulk copies on one mbarrier)
  float acc[kRtTok];
#pragma unroll
  for (int t = 0; t < kRtTok; ++t) acc[t] = 0.f;
  for (int c0 = 0, ch = 0; c0 < H; c0 += hc, ++ch) {
    const int len = min(hc, H - c0);
    if (tid == 0) {
      const uint32_t xbytes = ch == 0 ? (uint32_t)(nt * H * 2) : 0u;
      mbar_arrive_expect_tx(b, xbytes + (uint32_t)(ne * len * 4));
      if (ch == 0) bulk_g2s(smem_u32(xs), a.x + (size_t)t0 * H, xbytes, b);
      for (int r = 0; r < ne; ++r)
        bulk_g2s(smem_u32(ws + r * hc), a.lay.Wr + (size_t)(e0 + r) * H + c0, (uint32_t)(len * 4), b);
    }
    // bounded wait; on expiry the error is recorded (PW_ERR_TIMEOUT on the host) and the
    // copies get one more bounded wait before the CTA goes on with whatever landed
    bool landed = false;
    for (int round = 0; round < 2 && !landed; ++round) {
      for (long i = 0; i < kRtSpin && !landed; ++i) landed = mbar_try_wait(b, (uint32_t)(ch & 1));
      if (!landed && round == 0 && tid == 0 && a.s.err) atomicOr(a.s.err, 2);
    }
    if (ch == 0) {
      // unit-gain RMSNorm of the layer input (PW_PRENORM): one warp per staged token
      if (warp < nt) {
        float ss = 0.f;
        // the shared-expert gate goes to the last expert group, which holds the fewest experts
        const float *wsg = blockIdx.y == gridDim.y - 1 ? a.lay.wsg : nullptr;
        float gz = 0.f;
        for (int h = lane * 2; h < H; h += 64) {
          const uint32_t v = *reinterpret_cast<const uint32_t *>(xs + warp * H + h);
          const float a0 = bf16f(v & 0xFFFF), a1 = bf16f(v >> 16);
          ss = fmaf(a0, a0, fmaf(a1, a1, ss));
          if (wsg) {
            const float2 g = *reinterpret_cast<const float2 *>(wsg + h);
            gz = fmaf(a0, g.x, fmaf(a1, g.y, gz));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ss += __shfl_xor_sync(0xffffffffu, ss, o);
          gz += __shfl_xor_sync(0xffffffffu, gz, o);
        }
        const float inv = (a.flags & 2) ? rsqrtf(ss / (float)H + 1e-6f) : 1.0f;
        if (lane == 0) {
          s_inv[warp] = inv;
          if (blockIdx.y == 0) a.s.inv_rms[t0 + warp] = inv;
          // the gate reads the layer input as the experts do (normalised under PW_PRENORM)
          if (wsg) a.s.sgate[t0 + warp] = 1.f / (1.f + expf(-gz * inv));
          if (blockIdx.y == 0) a.s.xnorm[t0 + warp] = sqrtf(ss) * inv;
        }
      }
      {  // the experts' fp16 input rows, a slice of 8-column vectors per expert group
        __syncthreads();
        const int nv = H / 8, per = (nv + gridDim.y - 1) / gridDim.y;
        const int v0 = blockIdx.y * per, wid = min(nv, v0 + per) - v0;
        for (int v = tid; v < nt * wid; v += kRtThreads) {
          const int t = v / wid, c = (v0 + v % wid) * 8;
          const uint4 raw = *reinterpret_cast<const uint4 *>(xs + t * H + c);
          const float inv = s_inv[t];
          const uint32_t r[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t o[4];
          bool fin = true;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float lo = bf16f(r[i]) * inv, hi = bf16f(r[i] >> 16) * inv;
            fin = fin && fp16_finite(lo) && fp16_finite(hi);
            o[i] = pack2(f2h(lo), f2h(hi));
          }
          if (!fin && a.s.err) atomicOr(a.s.err, kErrRange);
          *reinterpret_cast<uint4 *>(a.s.xh + (size_t)(t0 + t) * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (a.s.ready) {  // publish the slice: the gate_up kernel reads it with tensor copies
          fence_proxy_async_global();
          __threadfence();
          __syncthreads();
          if (tid == 0) atomicAdd(a.s.ready + 2 * a.layer, 1);
        }
      }
    }
    if (warp < ne) {
      const float *wr = ws + warp * hc;
#pragma unroll 4
      for (int h = lane * 4; h < len; h += 128) {
        const float4 wv = *reinterpret_cast<const float4 *>(wr + h);
#pragma unroll
        for (int t = 0; t < kRtTok; ++t) {
          const uint2 xv = *reinterpret_cast<const uint2 *>(xs + t * H + c0 + h);
          acc[t] = fmaf(bf16f(xv.x & 0xFFFF), wv.x, acc[t]);
          acc[t] = fmaf(bf16f(xv.x >> 16), wv.y, acc[t]);
          acc[t] = fmaf(bf16f(xv.y & 0xFFFF), wv.z, acc[t]);
          acc[t] = fmaf(bf16f(xv.y >> 16), wv.w, acc[t]);
        }
      }
    }
    __syncthreads();  // the chunk buffer is rewritten by the next copy
  }
  if (warp < ne) {
    const float bias = a.lay.bias ? a.lay.bias[e0 + warp] : 0.f;
#pragma unroll
    for (int t = 0; t < kRtTok; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t < nt) a.s.logits[(size_t)(t0 + t) * E + e0 + warp] = v * s_inv[t] + bias;
    }
  }

  // ---- the last expert group of this token group ranks its tokens
  __threadfence();
  __syncthreads();
  unsigned *group_ticket = a.s.ticket + 1 + blockIdx.x;
  if (tid == 0) s_flag = atomicAdd(group_ticket, 1u) == gridDim.y - 1;
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  if (warp < nt) softmax_topk_warp(a, t0 + warp, lane);
  if (tid == 0) *group_ticket = 0u;

  // ---- the last token group buckets every pair
  __threadfence();
  __syncthreads();
  if (tid == 0) s_flag = atomicAdd(a.s.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_flag) return;
  __threadfence();

  const int T = a.T, TK = T * K;
  const RouteSmem rs = route_smem(T, K, H);
  int *s_ids = reinterpret_cast<int *>(smem_raw);
  float *s_w = reinterpret_cast<float *>(smem_raw) + TK;
  // a load whose latency overlaps the bucketing: the committed bitwidths of the layer's blocks
  const BlockDev *tab = a.table + (size_t)a.layer * E * 2;
  const int q1 = tid < E ? tab[2 * tid].q : 0, q2 = tid < E ? tab[2 * tid + 1].q : 0;
  if (rs.pairs) {  // the pairs were written by other CTAs: read them through L2
    for (int j0 = 0; j0 < TK; j0 += 4 * kRtThreads) {
      int iv[4];
      float wv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * kRtThreads + tid;
        iv[u] = j < TK ? __ldcg(a.s.ids + j) : 0;
        wv[u] = j < TK ? __ldcg(a.s.w + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * kRtThreads + tid;
        if (j < TK) {
          s_ids[j] = iv[u];
          s_w[j] = wv[u];
        }
      }
    }
  }
  const int *pid = rs.pairs ? s_ids : a.s.ids;
  const float *pwt = rs.pairs ? s_w : a.s.w;

  // bucketing: pair j = (t, k) goes to slot offsets[e] + (rank of j among expert e's pairs)
  __shared__ int s_wc[kRtWarps][256];  // per warp and expert: pairs counted, then first rank
  __shared__ int s_off[257];
  __shared__ int s_itm1[257];
  __shared__ int s_itm2[257];
  __shared__ int s_q[2][256];  // bitwidths, then item counts by rank
  __shared__ int s_rk[2][256];  // expert of each rank
  __shared__ int s_wsum[3][kRtWarps];
  for (int i = tid; i < kRtWarps * 256; i += kRtThreads) (&s_wc[0][0])[i] = 0;
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  const int span = (TK + kRtWarps - 1) / kRtWarps;
  const int j0 = warp * span, j1 = min(TK, j0 + span);
  // each warp walks its span 32 pairs at a time, with the loads of four batches in flight;
  // lanes past the span hold -1 - lane, which matches no expert and no other lane
  for (int jb = j0; jb < j1; jb += 4 * 32) {
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = jb + 32 * u + lane;
      ev[u] = j < j1 ? (rs.pairs ? pid[j] : __ldcg(pid + j)) : -1 - lane;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (jb + 32 * u >= j1) break;  // warp-uniform
      const unsigned peers = __match_any_sync(0xffffffffu, ev[u]);
      if (ev[u] >= 0 && (peers & lt) == 0u) s_wc[warp][ev[u]] += __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();
  const int tiles1 = (2 * a.I + kCtaRows - 1) / kCtaRows;
  const int tiles2 = (a.H + kCtaRows - 1) / kCtaRows;
  const int tc = tok_chunk_for(T);
  const int sh1 = shared_item_count(0, T, a.H, a.I, a.Is);
  const int sh2 = shared_item_count(1, T, a.H, a.I, a.Is);
  {
    int cnt = 0;
    if (tid < E)
      for (int w = 0; w < kRtWarps; ++w) {
        const int c = s_wc[w][tid];
        s_wc[w][tid] = cnt;
        cnt += c;
      }
    const int ch = (cnt + tc - 1) / tc;
    // The routed work items of the experts are laid out by decreasing committed bitwidth
    // (ties by expert id), separately for the two projections: an item's time grows with its
    // bitwidth, and items are claimed in list order, so the longest go first and the tail of
    // the launch is made of the shortest.
    if (tid < E) {
      s_q[0][tid] = q1;
      s_q[1][tid] = q2;
    }
    __syncthreads();
    int r1 = 0, r2 = 0;  // ranks in the two orders
    if (tid < E)
#pragma unroll 8
      for (int e = 0; e < E; ++e) {
        r1 += s_q[0][e] > q1 || (s_q[0][e] == q1 && e < tid);
        r2 += s_q[1][e] > q2 || (s_q[1][e] == q2 && e < tid);
      }
    __syncthreads();
    if (tid < E) {  // item counts in rank order (the q table is no longer needed)
      s_q[0][r1] = ch * tiles1;
      s_q[1][r2] = ch * tiles2 * routed_down_splits(T, a.I);
      s_rk[0][r1] = tid;
      s_rk[1][r2] = tid;
    }
    __syncthreads();
    int x0 = cnt, x1 = tid < E ? s_q[0][tid] : 0, x2 = tid < E ? s_q[1][tid] : 0;  // inclusive scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, x0, o);
      const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
      const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
      if (lane >= o) {
        x0 += y0;
        x1 += y1;
        x2 += y2;
      }
    }
    if (lane == 31) {
      s_wsum[0][warp] = x0;
      s_wsum[1][warp] = x1;
      s_wsum[2][warp] = x2;
    }
    __syncthreads();
    for (int w = 0; w < warp; ++w) {
      x0 += s_wsum[0][w];
      x1 += s_wsum[1][w];
      x2 += s_wsum[2][w];
    }
    if (tid < E) {  // exclusive scans in rank order, by rank
      s_off[tid] = x0 - cnt;
      s_itm1[tid] = sh1 + x1 - s_q[0][tid];
      s_itm2[tid] = sh2 + x2 - s_q[1][tid];
    }
    if (tid == kRtThreads - 1) {
      s_off[E] = x0;
      s_itm1[E] = sh1 + x1;
      s_itm2[E] = sh2 + x2;
    }
  }
  __syncthreads();
  for (int i = tid; i <= E; i += kRtThreads) a.s.offsets[i] = s_off[i];
  if (tid == 0) {
    a.s.n_items[0] = s_itm1[E];
    a.s.n_items[1] = s_itm2[E];
  }
  for (int jb = j0; jb < j1; jb += 4 * 32) {
    int ev[4];
    float wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = jb + 32 * u + lane;
      const bool in = j < j1;
      ev[u] = in ? (rs.pairs ? pid[j] : __ldcg(pid + j)) : -1 - lane;
      wv[u] = in ? (rs.pairs ? pwt[j] : __ldcg(pwt + j)) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (jb + 32 * u >= j1) break;  // warp-uniform
      const int j = jb + 32 * u + lane, ee = ev[u];
      const unsigned peers = __match_any_sync(0xffffffffu, ee);
      if (ee >= 0) {
        const int slot = s_off[ee] + s_wc[warp][ee] + __popc(peers & lt);
        a.s.slot_tok[slot] = j / K;
        a.s.pair_slot[j] = slot;
        a.s.slot_w[slot] = wv[u];
      }
      __syncwarp();
      if (ee >= 0 && (peers & lt) == 0u) s_wc[warp][ee] += __popc(peers);
      __syncwarp();
    }
  }
  // the work-list tables (the gather kernel that follows writes the work items from them)
  if (a.s.ranks)
    for (int i = tid; i <= E; i += kRtThreads) {
      a.s.ranks[i] = s_itm1[i];
      a.s.ranks[kRankStride + i] = s_itm2[i];
      if (i < E) {
        a.s.ranks[2 * kRankStride + i] = s_rk[0][i];
        a.s.ranks[3 * kRankStride + i] = s_rk[1][i];
      }
    }
  if (tid == 0) *a.s.ticket = 0u;
}

int launch_route(const FwdArgs &a, void *stream_) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_);
  const RouteSmem rs = route_smem(a.T, a.K, a.H);
  if (rs.bytes > kRtMaxSmem) return (int)cudaErrorInvalidValue;
  cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtMaxSmem);
  dim3 rg((a.T + kRtTok - 1) / kRtTok, (a.E + kRtExp - 1) / kRtExp);
  return (int)launch_pdl(route_kernel, rg, dim3(kRtThreads), (size_t)rs.bytes, st, a);
}

}  // namespace pw
