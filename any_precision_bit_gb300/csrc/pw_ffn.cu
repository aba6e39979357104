// pw_ffn.cu -- the expert kernels of the fused mixed-precision MoE layer (sm_103a).
//
// PagedWeight Sec. 3.3: every active expert's linear block is read directly from its
// bit-planes and LUT at its committed bitwidth q_i (Sec. 3.1 weight page table), the gate_up
// output goes through SiLU(gate)*up ("expert activation"), and the down projection follows.
// The shared expert of the layer (Table 1) rides in the same launches.
//
// One persistent CTA per SM, warp-specialised:
//   * warp 8 (producer) walks the CTA's work items and fills a ring of shared-memory stages.
//     Each stage is one 128-column chunk of a 128-row CTA tile: the q bit-planes (or the
//     fp16 shared weights) arrive by TMA bulk copies (cp.async.bulk, one per plane, each a
//     contiguous run thanks to the kernel-private tiling), the tokens' fp16 activation rows
//     by 16-byte cp.async gathers.  Both complete on the stage's "full" mbarrier.  The
//     tile's LUT_q rows arrive by one bulk copy per item on a separate barrier pair.
//   * warps 0..7 (consumers) each own a 16-row warp tile.  Per chunk a thread reads its one
//     word per plane per row, an 8x8 bit transpose yields the MSB-aligned codes of its
//     m16n8k16 A fragment, the codes index LUT_q in shared memory, and the fp16 centroids
//     go straight into the A registers; tokens are the N side (8 per MMA, up to 64 per
//     item).  A consumer releases the stage on its "empty" mbarrier.
// Every mbarrier wait is bounded: on expiry the kernel records an error (PW_ERR_TIMEOUT on
// the host), lets the producer wait for the copies it issued, and returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw_device.cuh"
#include "pw_internal.h"

namespace pw {

constexpr int kConsumers = kWarpsPerCta;              // 8 consumer warps
constexpr int kFfnThreads = (kConsumers + 1) * 32;    // + 1 producer warp
constexpr int kXRowBytes = (kChunkCols + 8) * 2;      // padded activation row: conflict-free B reads
constexpr int kPlaneStride = kWarpsPerCta * 256;      // bytes of one plane in a stage
constexpr int kFragStageBytes = 8 * kWarpsPerCta * 512;  // 8 steps of fp16 shared weights
constexpr long kSpinLimit = 1L << 22;
constexpr int kSmemLimit = 227 * 1024 - 1024;          // dynamic shared memory per CTA

struct FfnLayout {
  int stages;       // ring depth
  int stage_bytes;  // bytes per stage
  int x_off;        // activation rows inside a stage
  int xt;           // activation rows per stage (multiple of 8)
  int lut_off;      // LUT buffer
  int bar_off;      // mbarriers: full[S], empty[S], lut_full, lut_empty
  int smem;         // total dynamic shared memory
};

struct ItemView {
  bool routed;
  int q;         // routed: committed bitwidth
  int nchunks;   // 128-column stages
  int nwt;       // warp tiles in this CTA tile
  int NT;        // warp tiles of the block
  int KC;        // routed: 128-column chunks; shared: 16-column steps (KS)
  int Kc;        // activation columns
  int ntok;
  int row0;      // first activation row: routed slot (expert-sorted), shared token
  const BlockDev *bd;
  const uint16_t *W;  // shared weights
};

template <int PHASE>
__device__ __forceinline__ ItemView view_item(const FwdArgs &a, const WorkItem &w) {
  ItemView v;
  v.ntok = w.ntok;
  if (w.kind == 0) {
    v.routed = true;
    v.bd = &a.table[(a.layer * a.E + w.expert) * 2 + (PHASE - 1)];
    v.q = v.bd->q;
    v.NT = v.bd->N / 16;
    v.KC = v.bd->KC;
    v.nchunks = v.KC;
    v.Kc = v.bd->K;
    v.row0 = a.s.offsets[w.expert] + w.tok0;
    v.W = nullptr;
  } else {
    v.routed = false;
    v.bd = nullptr;
    v.q = 0;
    const int N = (PHASE == 1) ? 2 * a.Is : a.H;
    v.Kc = (PHASE == 1) ? a.H : a.Is;
    v.NT = N / 16;
    v.KC = v.Kc / 16;
    v.nchunks = (v.KC + 7) / 8;
    v.row0 = w.tok0;
    v.W = (PHASE == 1) ? a.lay.wgu : a.lay.wd;
  }
  v.nwt = cta_warps(w.tile, v.NT);
  return v;
}

// Activation row j of an item, fp16.
template <int PHASE>
__device__ __forceinline__ const uint16_t *act_row(const FwdArgs &a, const ItemView &v, int j) {
  if (PHASE == 1) {
    const int t = v.routed ? a.s.slot_tok[v.row0 + j] : v.row0 + j;
    return a.s.xh + (size_t)t * a.H;
  }
  return v.routed ? a.s.h_routed + (size_t)(v.row0 + j) * a.I : a.s.h_shared + (size_t)(v.row0 + j) * a.Is;
}

// LUT buffer: 512-byte aligned inside the dynamic shared memory (same for producer and consumers)
__device__ __forceinline__ uint32_t lut_base(const uint8_t *sm, const FfnLayout &L) {
  return (smem_u32(sm) + L.lut_off + 511u) & ~511u;
}

// Bounded wait on an mbarrier phase; false on expiry or when another warp gave up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *err) {
  for (long i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  atomicExch(err, 1);
  return false;
}

// ------------------------------------------------------------------ producer warp
template <int PHASE>
__device__ void producer(const FwdArgs &a, const FfnLayout &L, uint8_t *sm, uint32_t bars,
                         volatile int *abort_flag) {
  const int lane = threadIdx.x & 31;
  const int S = L.stages;
  const uint32_t full0 = bars, empty0 = bars + 8 * S, lut_full = bars + 16 * S, lut_empty = lut_full + 8;
  const int n_items = a.s.n_items[PHASE - 1];
  const WorkItem *items = (PHASE == 1) ? a.s.items1 : a.s.items2;
  uint32_t stage_seq = 0, lut_seq = 0;
  bool ok = true;
  for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
    const WorkItem w = items[it];
    const ItemView v = view_item<PHASE>(a, w);
    const int rt0 = w.tile * kWarpsPerCta;
    if (v.routed) {
      if (lane == 0) {
        ok = wait_bar(lut_empty, (lut_seq & 1) ^ 1, abort_flag, a.s.err);
        if (ok) {
          const uint32_t bytes = (uint32_t)(v.nwt * 16) << v.q << 1;
          mbar_arrive_expect_tx(lut_full, bytes);
          bulk_g2s(lut_base(sm, L), v.bd->lut[v.q] + ((size_t)rt0 * 16 << v.q), bytes, lut_full);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++lut_seq;
    }
    // this lane's activation rows (lane, lane + 32): base addresses once per item
    const uint16_t *rb0 = lane < v.ntok ? act_row<PHASE>(a, v, lane) : nullptr;
    const uint16_t *rb1 = lane + 32 < v.ntok ? act_row<PHASE>(a, v, lane + 32) : nullptr;
    for (int kc = w.kc0; kc < w.kc1 && ok; ++kc, ++stage_seq) {
      const int s = stage_seq % S;
      const uint32_t ph = (stage_seq / S) & 1;
      uint8_t *st = sm + (size_t)s * L.stage_bytes;
      if (lane == 0) ok = wait_bar(empty0 + 8 * s, ph ^ 1, abort_flag, a.s.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t full = full0 + 8 * s;
      if (lane == 0) {
        if (v.routed) {
          const uint32_t bytes = (uint32_t)v.nwt * 256;
          mbar_arrive_expect_tx(full, bytes * v.q);
          const long off = plane_pair_word(rt0, kc, v.NT, v.KC);
          for (int p = 0; p < v.q; ++p)
            bulk_g2s(smem_u32(st + p * kPlaneStride), v.bd->plane[p] + off, bytes, full);
        } else {
          const int nks = min(8, v.KC - kc * 8);
          const uint32_t bytes = (uint32_t)(nks * v.nwt) * 512;
          mbar_arrive_expect_tx(full, bytes);
          bulk_g2s(smem_u32(st), v.W + 2 * frag_pair_word(rt0, kc * 8, v.NT, v.KC), bytes, full);
        }
      }
      const uint32_t xdst = smem_u32(st + L.x_off);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int j = lane + 32 * r;
        if (j >= L.xt) break;
        const uint16_t *rb = r ? rb1 : rb0;
#pragma unroll 4
        for (int c16 = 0; c16 < 16; ++c16) {
          const int col = kc * kChunkCols + c16 * 8;
          const bool valid = rb != nullptr && col < v.Kc;
          cp_async16(xdst + j * kXRowBytes + c16 * 16, valid ? rb + col : a.s.xh, valid ? 16u : 0u);
        }
      }
      cp_async_arrive(full);
    }
  }
  // every copy this warp issued must land before the CTA may exit
  if (lane == 0) {
    for (uint32_t k = 0; k < (uint32_t)S && k < stage_seq; ++k) {
      const uint32_t q = stage_seq - 1 - k;
      for (long i = 0; i < kSpinLimit && !mbar_try_wait(full0 + 8 * (q % S), (q / S) & 1); ++i) {
      }
    }
    if (lut_seq > 0)
      for (long i = 0; i < kSpinLimit && !mbar_try_wait(lut_full, (lut_seq - 1) & 1); ++i) {
      }
  }
}

// ------------------------------------------------------------------ consumer warps
template <int PHASE, bool SHARED>
__device__ __forceinline__ void epilogue(const FwdArgs &a, const ItemView &v, int rt, int ngroups,
                                         float (&acc)[8][4], int part) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= ngroups) break;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int tj = 8 * j + 2 * c + h;
      if (tj >= v.ntok) continue;
      if (PHASE == 1) {
        const int f = rt * 8 + g;
        const float hv = silu(acc[j][h]) * acc[j][2 + h];
        if (SHARED)
          a.s.h_shared[(size_t)(v.row0 + tj) * a.Is + f] = f2h(hv);
        else
          a.s.h_routed[(size_t)(v.row0 + tj) * a.I + f] = f2h(hv);
      } else {
        const int r0 = rt * 16 + g;
        float *dst = SHARED ? a.s.o_shared + ((size_t)part * a.T + v.row0 + tj) * a.H
                            : a.s.o_routed + (size_t)(v.row0 + tj) * a.H;
        dst[r0] = acc[j][h];
        dst[r0 + 8] = acc[j][2 + h];
      }
    }
  }
}

// ldmatrix row address of this thread for B fragments: matrices (group j, k 0-7), (j, k 8-15),
// (j+1, k 0-7), (j+1, k 8-15) of a 16-column step; rows are tokens.
__device__ __forceinline__ uint32_t b_lane_offset() {
  const int lane = threadIdx.x & 31;
  return (uint32_t)(((((lane >> 4) & 1) * 8 + (lane & 7)) * kXRowBytes) + ((lane >> 3) & 1) * 16);
}

// B fragments of all token groups of one 16-column step, two groups per ldmatrix.
template <int NG>
__device__ __forceinline__ void load_b_step(uint32_t xs_lane, int s, uint32_t (&b)[8][2]) {
#pragma unroll
  for (int j = 0; j < NG; j += 2) {
    const uint32_t addr = xs_lane + j * 8 * kXRowBytes + s * 32;
    if (j + 1 < NG)
      ldm_x4(addr, b[j][0], b[j][1], b[j + 1][0], b[j + 1][1]);
    else
      ldm_x2(addr, b[j][0], b[j][1]);
  }
}

// Shared-memory address of LUT entry `code` of a row whose table starts at a base aligned to
// 2^(Q+1) bytes: the code, shifted to bytes, is OR-ed into the base.  Y holds MSB-aligned
// codes in its bytes; E selects the byte.
template <int Q, int E>
__device__ __forceinline__ uint32_t lut_addr(uint32_t Y, uint32_t base) {
  constexpr int sh = 8 * E + 7 - Q;
  constexpr uint32_t m = ((1u << Q) - 1u) << 1;
  const uint32_t v = sh >= 0 ? (Y >> (sh >= 0 ? sh : 0)) : (Y << (sh < 0 ? -sh : 0));
  return (v & m) | base;
}

// The A-fragment register of elements (E, E+1) of row base `base` from code word Y.
template <int Q, int E>
__device__ __forceinline__ uint32_t lut_pair(uint32_t Y, uint32_t base) {
  return lds_pair(lut_addr<Q, E>(Y, base), lut_addr<Q, E + 1>(Y, base));
}

// One stage of a routed item at compile-time group count NG.
template <int Q, int NG>
__device__ __forceinline__ void routed_stage(const uint8_t *st, uint32_t xs_lane, uint32_t lg, uint32_t l8,
                                             float (&acc)[8][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint2 pw_[Q];
#pragma unroll
  for (int p = 0; p < Q; ++p)
    pw_[p] = *reinterpret_cast<const uint2 *>(st + p * kPlaneStride + warp * 256 + lane * 8);
  uint32_t Yg[8], Y8[8];
  codes_from_planes<Q>(pw_, Yg, Y8);
#pragma unroll
  for (int s8 = 0; s8 < 8; ++s8) {
    const uint32_t a0 = lut_pair<Q, 0>(Yg[s8], lg);
    const uint32_t a1 = lut_pair<Q, 0>(Y8[s8], l8);
    const uint32_t a2 = lut_pair<Q, 2>(Yg[s8], lg);
    const uint32_t a3 = lut_pair<Q, 2>(Y8[s8], l8);
    uint32_t b[8][2];
    load_b_step<NG>(xs_lane, s8, b);
#pragma unroll
    for (int j = 0; j < NG; ++j) mma_f16(acc[j], a0, a1, a2, a3, b[j][0], b[j][1]);
  }
}

// Returns false when a wait gave up.
template <int PHASE, int Q>
__device__ bool routed_item(const FwdArgs &a, const FfnLayout &L, uint8_t *sm, uint32_t bars,
                            volatile int *abort_flag, const ItemView &v, const WorkItem &w,
                            uint32_t &stage_seq, uint32_t &lut_seq) {
  const int tile = w.tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2;
  const int S = L.stages;
  const uint32_t full0 = bars, empty0 = bars + 8 * S, lut_full = bars + 16 * S, lut_empty = lut_full + 8;
  const bool active = warp < v.nwt;
  const int rt = tile * kWarpsPerCta + warp;
  const int ngroups = (v.ntok + 7) / 8;
  const uint32_t lg = lut_base(sm, L) + ((uint32_t)(warp * 16 + g) << (Q + 1));
  const uint32_t l8 = lg + (8u << (Q + 1));
  const uint32_t xoff = (uint32_t)L.x_off + b_lane_offset();
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
  if (!wait_bar(lut_full, lut_seq & 1, abort_flag, a.s.err)) return false;
  for (int kc = w.kc0; kc < w.kc1; ++kc, ++stage_seq) {
    const int s = stage_seq % S;
    if (!wait_bar(full0 + 8 * s, (stage_seq / S) & 1, abort_flag, a.s.err)) return false;
    const uint8_t *st = sm + (size_t)s * L.stage_bytes;
    if (active) {
      const uint32_t xs_lane = smem_u32(st) + xoff;
      switch (ngroups) {
        case 1: routed_stage<Q, 1>(st, xs_lane, lg, l8, acc); break;
        case 2: routed_stage<Q, 2>(st, xs_lane, lg, l8, acc); break;
        case 3: case 4: routed_stage<Q, 4>(st, xs_lane, lg, l8, acc); break;
        default: routed_stage<Q, 8>(st, xs_lane, lg, l8, acc); break;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(lut_empty);
  ++lut_seq;
  if (active) epilogue<PHASE, false>(a, v, rt, ngroups, acc, 0);
  return true;
}

template <int NG>
__device__ __forceinline__ void shared_stage(const uint8_t *st, uint32_t xs_lane, int nks, int nwt,
                                             float (&acc)[8][4]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int ks = 0; ks < nks; ++ks) {
    const uint4 af = *reinterpret_cast<const uint4 *>(st + (ks * nwt + warp) * 512 + lane * 16);
    uint32_t b[8][2];
    load_b_step<NG>(xs_lane, ks, b);
#pragma unroll
    for (int j = 0; j < NG; ++j) mma_f16(acc[j], af.x, af.y, af.z, af.w, b[j][0], b[j][1]);
  }
}

template <int PHASE>
__device__ bool shared_item(const FwdArgs &a, const FfnLayout &L, uint8_t *sm, uint32_t bars,
                            volatile int *abort_flag, const ItemView &v, const WorkItem &w,
                            uint32_t &stage_seq) {
  const int tile = w.tile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = L.stages;
  const uint32_t full0 = bars, empty0 = bars + 8 * S;
  const bool active = warp < v.nwt;
  const int rt = tile * kWarpsPerCta + warp;
  const int ngroups = (v.ntok + 7) / 8;
  const uint32_t xoff = (uint32_t)L.x_off + b_lane_offset();
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
  for (int kc = w.kc0; kc < w.kc1; ++kc, ++stage_seq) {
    const int s = stage_seq % S;
    if (!wait_bar(full0 + 8 * s, (stage_seq / S) & 1, abort_flag, a.s.err)) return false;
    const uint8_t *st = sm + (size_t)s * L.stage_bytes;
    if (active) {
      const int nks = min(8, v.KC - kc * 8);
      const uint32_t xs_lane = smem_u32(st) + xoff;
      switch (ngroups) {
        case 1: shared_stage<1>(st, xs_lane, nks, v.nwt, acc); break;
        case 2: shared_stage<2>(st, xs_lane, nks, v.nwt, acc); break;
        case 3: case 4: shared_stage<4>(st, xs_lane, nks, v.nwt, acc); break;
        default: shared_stage<8>(st, xs_lane, nks, v.nwt, acc); break;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
  if (active) epilogue<PHASE, true>(a, v, rt, ngroups, acc, w.part);
  return true;
}

template <int PHASE>
__device__ void consumer(const FwdArgs &a, const FfnLayout &L, uint8_t *sm, uint32_t bars,
                         volatile int *abort_flag) {
  const int n_items = a.s.n_items[PHASE - 1];
  const WorkItem *items = (PHASE == 1) ? a.s.items1 : a.s.items2;
  uint32_t stage_seq = 0, lut_seq = 0;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const WorkItem w = items[it];
    const ItemView v = view_item<PHASE>(a, w);
    bool ok;
    if (!v.routed) {
      ok = shared_item<PHASE>(a, L, sm, bars, abort_flag, v, w, stage_seq);
    } else {
      switch (v.q) {
        case 1: ok = routed_item<PHASE, 1>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
        case 2: ok = routed_item<PHASE, 2>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
        case 3: ok = routed_item<PHASE, 3>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
        case 4: ok = routed_item<PHASE, 4>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
        case 5: ok = routed_item<PHASE, 5>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
        case 6: ok = routed_item<PHASE, 6>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
        case 7: ok = routed_item<PHASE, 7>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
        default: ok = routed_item<PHASE, 8>(a, L, sm, bars, abort_flag, v, w, stage_seq, lut_seq); break;
      }
    }
    if (!ok) return;
  }
}

template <int PHASE>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_kernel(FwdArgs a, FfnLayout L) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ int abort_flag;
  const uint32_t bars = smem_u32(sm + L.bar_off);
  if (threadIdx.x == 0) {
    for (int s = 0; s < L.stages; ++s) {
      mbar_init(bars + 8 * s, 33);                             // full: 1 expect_tx + 32 cp.async lanes
      mbar_init(bars + 8 * (L.stages + s), kConsumers);        // empty: one arrival per consumer warp
    }
    mbar_init(bars + 16 * L.stages, 1);                        // lut_full
    mbar_init(bars + 16 * L.stages + 8, kConsumers);           // lut_empty
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == kConsumers)
    producer<PHASE>(a, L, sm, bars, &abort_flag);
  else
    consumer<PHASE>(a, L, sm, bars, &abort_flag);
}

static FfnLayout ffn_layout(const FwdArgs &a, int bmax_lut_entries) {
  FfnLayout L{};
  const int wbytes = a.Is > 0 ? kFragStageBytes : kMaxPlanes * kPlaneStride;
  // activation rows per stage: the token groups rounded the way the consumers round them
  // (1, 2, 4 or 8 groups of 8), so that every row an ldmatrix reads lies in the stage
  const int groups = (min(a.T, kTokChunk) + 7) / 8;
  L.xt = 8 * (groups <= 2 ? groups : (groups <= 4 ? 4 : 8));
  L.x_off = wbytes;
  L.stage_bytes = (wbytes + L.xt * kXRowBytes + 127) / 128 * 128;
  const int lut_bytes = kCtaRows * bmax_lut_entries * 2 + 512;  // + alignment slack
  const int budget = kSmemLimit - lut_bytes - 256;
  L.stages = min(6, budget / L.stage_bytes);
  L.lut_off = L.stages * L.stage_bytes;
  L.bar_off = L.lut_off + lut_bytes;
  L.smem = L.bar_off + (2 * L.stages + 2) * 8;
  return L;
}

int launch_ffn(const FwdArgs &a, int phase, void *stream) {
  const FfnLayout L = ffn_layout(a, 256);
  if (L.stages < 2) return (int)cudaErrorInvalidConfiguration;
  static int attr_done = 0;
  if (!attr_done) {
    cudaFuncSetAttribute(ffn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    cudaFuncSetAttribute(ffn_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    attr_done = 1;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int max_items = phase == 1 ? a.s.max_items1 : a.s.max_items2;
  const int grid = min(max_items, a.sm_count);
  if (phase == 1)
    ffn_kernel<1><<<grid, kFfnThreads, L.smem, st>>>(a, L);
  else
    ffn_kernel<2><<<grid, kFfnThreads, L.smem, st>>>(a, L);
  return (int)cudaGetLastError();
}

}  // namespace pw
