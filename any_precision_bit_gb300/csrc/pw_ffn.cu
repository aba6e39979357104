// pw_ffn.cu -- the expert kernels of the fused mixed-precision MoE layer on the 5th-generation
// tensor cores (sm_103a).
//
// PagedWeight Sec. 3.3: every active expert's linear block is read directly from its
// bit-planes and LUT at its committed bitwidth q_i (Sec. 3.1 weight page table), the gate_up
// output goes through the expert activation SiLU(gate)*up, and the down projection follows.
// The shared expert of the layer (Table 1) rides in the same launches.
//
// A work item is a 128-row tile of one block times up to TOK tokens: D[128][N] = W x X^T,
// N = tokens padded to 16, accumulated in tensor memory.  TOK = 64 at decode batch sizes; for
// prefill-sized batches TOK = 128, so that each dequantised weight tile feeds twice the
// tokens (the accumulators then fill half of tensor memory, and the activation tiles are
// split along K into two 64-column stages to fit shared memory).  One persistent CTA per SM,
// warp-specialised:
//   * LUT producer (1 warp): per routed item the tile's LUT_q rows (one TMA bulk copy) into
//     one of two LUT slots, so that the next item's table loads while this one runs (a q = 8
//     table takes both);
//   * weight producer (1 warp): claims the work items one at a time from the launch's atomic
//     counter when it is ready to stream the next one (so CTAs that finish early take more),
//     publishes them in order to the other roles through a shared-memory queue, and copies
//     per 128-column chunk the weights into a ring of 2 KB slabs:
//     the q bit-plane slabs of a routed chunk (lane p copies plane p) or the eight 4 KB K-step
//     pieces of a dense shared-expert tile (lane t copies piece t).  A chunk takes exactly the
//     bytes it needs, so low bitwidths keep more chunks in flight.  A routed chunk's slabs
//     return to the ring once its dequantising warps have read them; the copies stream with
//     an L2 evict-first policy (except a prefill gate_up, whose tiles several token chunks
//     read), so that the activations stay in L2;
//   * activation producer (1 warp): the B operand tiles, three per-chunk slots of two stages
//     (64 columns each, 128-byte swizzle), loaded by TMA from row-contiguous buffers (the
//     layer input gathered into slot order beforehand, h, the shared expert's input and h):
//     decode, one 16-row box per lane, as many as the item has tokens padded to 16; prefill,
//     one 128-row box per stage.  TMA keeps every slot's copies in flight at once (16-byte
//     cp.async gathers stall on one round trip per tile);
//   * dequantising warps (16: four chunk streams, each with one warp per tensor-memory lane
//     quarter): stream s takes the routed chunks c with c mod 4 = s; each thread owns one row
//     and the chunk's 128 columns, turns its plane words into fp16 centroids (pw_dq.cuh) and
//     writes them straight into tensor memory (tcgen05.st), a 4-deep ring of A buffers, so
//     that one stream's store wait overlaps the others' arithmetic.  In the GEMV kernel image
//     they also compute small routed items on the CUDA cores (below the GEMV threshold);
//   * MMA warp (1 warp): per chunk eight tcgen05.mma (M = 128, N, K = 16), issued by one
//     elected lane of the converged warp, with A read from tensor memory (routed blocks) or
//     from the slab ring (shared expert), B from shared memory, the accumulator in one of two
//     tensor-memory buffers; tcgen05.commit releases the A buffer, the B tile and a dense
//     chunk's slabs when the MMAs are done;
//   * epilogue (4 warps, one per lane quarter): tcgen05.ld of the accumulator, then
//     h = silu(g) * u (gate_up) or the down output, while the next item is being computed.
//     A down item that covers one K part (the shared expert's down, and at decode sizes a
//     long routed down) writes that part's partial-sum buffer; the combine kernel adds the
//     parts in order.
// The shared expert's items lead the work list and depend only on their activations: they
// start once the router has counted the layer's input rows ready (gate_up) or every shared
// gate_up item has counted its h written (down), while the routed items wait for the
// previous kernels to complete (griddepcontrol.wait).
// Every wait is bounded: on expiry the kernel records an error (PW_ERR_TIMEOUT on the host),
// every role stops, the producers and the MMA warp wait (bounded) for what they issued, and
// tensor memory is freed before the kernel returns.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pw_device.cuh"
#include "pw_dq.cuh"
#include "pw_internal.h"
#include "pw_tc.cuh"

namespace pw {

// Routed work items of at most FwdArgs::gemv_max tokens (decode tiling) run on the CUDA cores
// (GEMV) instead of the tensor cores; kGemvMaxTok bounds that threshold.
constexpr int kGemvMaxTok = kGemvMaxTokens;
static_assert(kGemvMaxTok >= 1 && kGemvMaxTok <= 8, "GEMV items hold at most 8 tokens");
constexpr int kGxSlots = 4;                 // activation slots of the GEMV items: one per chunk stream
constexpr int kGxBytes = 8 * kChunkCols * 2;  // one slot: 8 rows x 128 fp16 columns
constexpr int kDqStreams = 4;               // chunk streams of dequantising warps
constexpr int kDq = 4 * kDqStreams;         // dequantising warps 0 .. 15 (warp w: lane quarter w & 3, stream w >> 2)
constexpr int kEpi = 4;                     // epilogue warps
constexpr int kWarpP = kDq + kEpi;          // weight producer
constexpr int kWarpAB = kWarpP + 1;         // activation producer
constexpr int kWarpMma = kWarpP + 2;        // MMA issuer, tensor-memory owner
constexpr int kWarpLut = kWarpP + 3;        // LUT producer
constexpr int kTcThreads = (kWarpLut + 1) * 32;
constexpr int kSlab = kCtaRows * 16;        // 2 KB: one plane of a 128-row tile and 128 columns
constexpr int kRing = 16;                   // chunks in flight (full/empty barrier pairs)
static_assert(kRing % kDqStreams == 0, "each barrier of the routed-chunk rings belongs to one chunk stream");
constexpr int kQueue = 8;                   // claimed work items published to the roles
constexpr int kQueueReaders = kDq + kEpi + 3;  // warps that read the queue (all but the weight producer)
constexpr int kAStagesMax = 6;              // tensor-memory A buffers (at most)
constexpr int kBStagesMax = 6;              // activation stages (at most)
constexpr int kDenseSlabs = 16;             // a dense 32 KB A tile: 8 pieces of 2 slabs
constexpr int kLutSlot = 32 * 1024;         // LUT slot (q <= 7); q = 8 takes both slots
constexpr int kACols = kChunkCols / 2;      // tensor-memory columns per A buffer (fp16 pairs)
constexpr uint32_t kTmemCols = 512;

// The token tiling of a launch.  Tensor memory: two accumulator buffers of TOK fp32 columns,
// then the kAStages A buffers (2 TOK + kAStages * 64 <= 512 columns).  Activation stages: TOK rows
// by 64 columns in the 128-byte swizzled K-major layout (8 KB or 16 KB), four MMA K-steps
// each; two stages make a chunk's slot.  kBLowStages of them sit below the LUT slots, the
// rest after them.
template <int TOK>
struct Tiling {
  static_assert(TOK == 64 || TOK == 128, "token tile");
  static constexpr int kAccCols = TOK;
  static constexpr uint32_t kAColBase = 2 * TOK;
  static constexpr int kBK = 64;                     // columns per stage: one 128-byte swizzle row
  static constexpr int kBPieces = kChunkCols / kBK;  // stages per chunk
  static constexpr int kBSteps = kBK / 16;           // MMA K-steps per stage
  static constexpr int kBStages = 6;
  static constexpr int kBSlots = kBStages / kBPieces;  // per-chunk slots (one full/empty barrier pair each)
  static constexpr int kBLowStages = TOK == 64 ? 6 : 3;
  static constexpr uint32_t kDescStep = 2u;  // descriptor start-address step (16 B units) of one K-step (32 B)
  static constexpr int kBoxRows = TOK == 64 ? 16 : 128;  // rows of one TMA box
  static constexpr int kAStages = TOK == 64 ? 4 : 4;
  static_assert(kAStages <= kAStagesMax && kAColBase + kAStages * kACols <= kTmemCols, "tensor memory");
  static_assert(kAStages % 4 == 0, "each A buffer belongs to one chunk stream");
  static_assert(kBStages <= kBStagesMax, "activation stages");
};
constexpr uint32_t kWaitSleepNs = 20000;  // suspend-time hint of a barrier wait
// The launch's wait limit in SM cycles (FwdArgs::wait_cycles), set by thread 0 before the
// roles start.
__shared__ long long s_wait_cycles;
constexpr int kSmemLimit = 227 * 1024 - 1024;

// Shared-memory map.  The host fills npad_max, b_bytes and smem (the dynamic size);
// the kernel places the regions by absolute shared address: the first kBLowStages
// activation stages, the GEMV items' activation slots and the mbarriers at the start of the
// dynamic area, the two LUT slots at
// [64 KB, 128 KB) (the tiled LUT layout needs a 64 KB-aligned table), then the other
// activation stages (prefill tiling), and the slab ring to the end.
struct TcLayout {
  int npad_max;    // B tile rows (tokens padded to 16)
  int b_bytes;     // one activation stage
  int smem;        // dynamic shared memory of the launch
  // filled in by the kernel, offsets from the dynamic area
  int slabs;       // slab ring size (even)
  int ring_off;    // slab ring
  int b_off;       // activation stages 0 .. kBLowStages - 1
  int b_hi;        // activation stages kBLowStages ..
  int lut_off;     // LUT slots
  int gx_off;      // activation slots of the GEMV items
  int bar_off;     // mbarriers
};
constexpr uint32_t kLutAddr = 64 * 1024;
constexpr uint32_t kRingAddr = 128 * 1024;

// mbarrier indices
enum {
  kWFR = 0, kWFD = kWFR + kRing, kWE = kWFD + kRing, kTAF = kWE + kRing, kTAE = kTAF + kAStagesMax, kBF = kTAE + kAStagesMax,
  kBE = kBF + kBStagesMax, kLF = kBE + kBStagesMax, kLE = kLF + 2, kAF = kLE + 2, kAE = kAF + 2, kDrain = kAE + 2,
  kIQF = kDrain + 1, kIQE = kIQF + kQueue, kGXF = kIQE + kQueue, kGXE = kGXF + kGxSlots, kGAG = kGXE + kGxSlots,
  kAFG = kGAG + 2, kRD = kAFG + 2, kNumBars = kRD + kRing
};

struct ItemView {
  bool routed;
  bool gemv;     // routed item of at most kGemvMaxTok tokens at the decode tiling: CUDA-core dot products
  int q;         // routed: committed bitwidth
  int nr;        // rows of this CTA tile
  int KC;        // 128-column chunks of the K dimension
  int Kc;        // activation columns
  int N;         // rows of the block
  int ntok, npad;
  int row0;      // first activation row: routed slot (expert-sorted), shared token
  const BlockDev *bd;
  const uint16_t *W;    // shared weights
  const uint16_t *lut;  // routed: LUT_q of the block (tiled layout)
};

template <int PHASE>
__device__ __forceinline__ ItemView view_item(const FwdArgs &a, const WorkItem &w) {
  ItemView v;
  v.ntok = w.ntok;
  v.npad = max(16, (w.ntok + 15) / 16 * 16);
  if (w.kind == 0) {
    v.routed = true;
    v.bd = &a.table[(a.layer * a.E + w.expert) * 2 + (PHASE - 1)];
    v.q = v.bd->q;
    v.N = v.bd->N;
    v.KC = v.bd->KC;
    v.Kc = v.bd->K;
    v.row0 = a.s.offsets[w.expert] + w.tok0;
    v.W = nullptr;
    v.lut = v.bd->lut[v.q];
    v.gemv = a.T < kPrefillMinT && w.ntok <= min(a.gemv_max, kGemvMaxTok);
  } else {
    v.routed = false;
    v.gemv = false;
    v.bd = nullptr;
    v.q = 0;
    v.N = (PHASE == 1) ? 2 * a.Is : a.H;
    v.Kc = (PHASE == 1) ? a.H : a.Is;
    v.KC = kpad_cols(v.Kc) / kChunkCols;
    v.row0 = w.tok0;
    v.W = (PHASE == 1) ? a.lay.wgu : a.lay.wd;
    v.lut = nullptr;
  }
  v.nr = tile_rows(w.tile, v.N);
  return v;
}

__device__ __forceinline__ uint32_t lut_base(const uint8_t *sm, const TcLayout &L) {
  return smem_u32(sm) + (uint32_t)L.lut_off;
}
template <int TOK>
__device__ __forceinline__ uint32_t b_stage(const uint8_t *sm, const TcLayout &L, int s) {
  constexpr int low = Tiling<TOK>::kBLowStages;
  return smem_u32(sm) + (uint32_t)(s < low ? L.b_off + s * L.b_bytes : L.b_hi + (s - low) * L.b_bytes);
}

// LUT slot schedule, replayed identically by the weight producer and the dequantising warps:
// tables of q <= 7 alternate between the two slots; a q = 8 table (64 KB) takes both.
struct LutSched {
  uint32_t fills[2] = {0u, 0u}, uses[2] = {0u, 0u};
  int last = 1;
  __device__ __forceinline__ int next(int q, bool &both) {
    both = q > 7;
    const int slot = both ? 0 : (last ^ 1);
    last = both ? 1 : slot;
    return slot;
  }
};

// Position in the slab ring, replayed identically by every role: chunk c (all items, in
// order) takes q consecutive slabs (routed; the ring's tail is skipped when they would wrap,
// so that the dequantising warps address the planes from one base) or 16 slabs starting at
// an even slab (dense; one padding slab when needed, so that no 4 KB piece wraps).  n = slabs consumed, padding included.
// Routed and dense chunks also count separately (seq): their "weights landed" barriers are
// separate sequences, because the dequantising warps wait only on routed chunks and skip
// the dense ones.  A waiter that skipped fills of a barrier could otherwise run two phases
// ahead of it, where a parity wait cannot tell the phase it wants from an old one.
struct RingPos {
  uint32_t slot = 0, c = 0, rc = 0, dc = 0;
  __device__ __forceinline__ uint32_t take(bool routed, int q, int S, uint32_t &n, uint32_t &seq) {
    uint32_t pad = routed ? 0u : (slot & 1u);
    const uint32_t nd = routed ? (uint32_t)q : (uint32_t)kDenseSlabs;
    uint32_t base = slot + pad;
    if (base >= (uint32_t)S) base -= (uint32_t)S;
    if (routed && base + nd > (uint32_t)S) {  // a routed chunk's planes never wrap: one base address
      pad += (uint32_t)S - base;
      base = 0;
    }
    slot = base + nd;
    if (slot >= (uint32_t)S) slot -= (uint32_t)S;
    n = pad + nd;
    seq = routed ? rc++ : dc++;
    ++c;
    return base;
  }
};
// "weights landed" barrier of a chunk: routed and dense sequences
__device__ __forceinline__ uint32_t wf_bar(uint32_t bars, bool routed, uint32_t seq) {
  return bars + 8 * ((routed ? kWFR : kWFD) + seq % kRing);
}
__device__ __forceinline__ uint32_t ring_add(uint32_t a, uint32_t b, int S) {
  const uint32_t r = a + b;
  return r >= (uint32_t)S ? r - (uint32_t)S : r;
}

// Bounded wait on an mbarrier phase; false on expiry or when another warp gave up.  A
// waiting thread sleeps in the barrier (suspend-time hint) rather than polling, so that it
// takes no issue slots from the warps it waits for; the bound is on elapsed SM clock cycles.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > s_wait_cycles) break;
  }
  *abort_flag = 1;
  atomicOr(err, 1);
  return false;
}
// Bounded wait for the inputs of the shared expert's items of this kernel: for gate_up the
// layer's fp16 input rows (every router CTA counted), for down the shared h (every epilogue
// warp of every shared gate_up item counted).  False on expiry or when another warp gave up.
// The shared items start on this instead of on the end of the previous kernels.
template <int PHASE>
__device__ __forceinline__ bool wait_ready(const FwdArgs &a, volatile int *abort_flag) {
  if (!a.s.ready) return true;
  const int *p = a.s.ready + 2 * a.layer + (PHASE - 1);
  const int target = PHASE == 1 ? route_ctas(a.T, a.E) : shared_item_count(0, a.T, a.H, a.I, a.Is) * kEpi;
  if (ld_acquire_gpu(p) >= target) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(200);
    if (ld_acquire_gpu(p) >= target) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > s_wait_cycles) break;
  }
  *abort_flag = 1;
  atomicOr(a.s.err, 1);
  return false;
}
// Wait that ignores the abort flag (used to drain what this thread issued); bounded.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kWaitSleepNs) && clock64() - t0 <= s_wait_cycles) {
  }
}
// Two waits taken by a whole warp; when both phases are already complete (the common case
// on the MMA warp) the two checks overlap their latencies.
__device__ __forceinline__ bool wait2_all(uint32_t b1, uint32_t p1, uint32_t b2, uint32_t p2, volatile int *abort_flag,
                                          int *err) {
  const bool r1 = mbar_try_wait(b1, p1);
  const bool r2 = mbar_try_wait(b2, p2);
  if (__all_sync(0xffffffffu, r1 && r2)) return true;
  return __all_sync(0xffffffffu, wait_bar(b1, p1, abort_flag, err) && wait_bar(b2, p2, abort_flag, err));
}
// The same wait taken by a whole warp, with one outcome for every lane.
__device__ __forceinline__ bool wait_bar_all(uint32_t bar, uint32_t parity, volatile int *abort_flag, int *err) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, err));
}

// Work items are claimed one at a time (atomic counter) by the weight producer and published,
// in order, in a shared-memory queue that every other role reads.  Entry k of a role's
// sequence holds the item index (-1 once the items are exhausted), the item, and the facts
// about it that every role needs; the producer reads them from global memory once, so that
// no other role waits on that latency.
struct QEntry {
  int it;
  WorkItem w;
  ItemView v;
};
struct ItemQueue {
  QEntry *slot;  // [kQueue]
  uint32_t bars;
};
// Reader side, one call per warp and entry (lane 0 releases the entry after the warp read it).
// `lanes`: the lanes of the warp that run the role (all, or lane 0 alone).  False once the
// items are exhausted (or on a timeout).
__device__ __forceinline__ bool queue_read(const ItemQueue &qu, uint32_t k, unsigned lanes, volatile int *abort_flag,
                                           int *err, WorkItem &w, ItemView &v) {
  bool ok = wait_bar(qu.bars + 8 * (kIQF + k % kQueue), (k / kQueue) & 1, abort_flag, err);
  if (lanes == 0xffffffffu) ok = __all_sync(0xffffffffu, ok);
  if (!ok) return false;
  const QEntry &e = qu.slot[k % kQueue];
  const int it = e.it;
  if (it >= 0) {
    w = e.w;
    v = e.v;
  }
  __syncwarp(lanes);
  if ((threadIdx.x & 31) == 0) mbar_arrive(qu.bars + 8 * (kIQE + k % kQueue));
  return it >= 0;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

// ------------------------------------------------------------------ roles
template <int PHASE>
__device__ void weight_producer(const FwdArgs &a, const TcLayout &L, uint8_t *sm, uint32_t bars,
                                const ItemQueue &qu, volatile int *abort_flag) {
  const int lane = threadIdx.x & 31;
  const WorkItem *items = (PHASE == 1) ? a.s.items1 : a.s.items2;
  const uint32_t ring = smem_u32(sm) + (uint32_t)L.ring_off;
  const int S = L.slabs;
  // The shared expert's items (the first n_shared of the list) need only their activations
  // (gate_up: the router's input rows; down: the shared h) and are built here; the routed
  // ones, the item count and the list wait for the previous kernels to complete.
  const int n_shared = shared_item_count(PHASE - 1, a.T, a.H, a.I, a.Is);
  int n_items = 0;
  bool routed_ready = false;
  // The weights are read once per launch at decode sizes, the activations by every row tile:
  // there the weights' lines go first.  A prefill gate_up tile is read by the several token
  // chunks of its expert, claimed together, and keeps the default policy (evict-first made
  // its DRAM reads 1.18x the algorithmic bytes instead of 1.05x).
  const uint64_t stream_policy = l2_evict_first_policy();
  const bool evict_first = PHASE == 2 || a.T < kPrefillMinT;
  RingPos pos;
  // room accounting (the same in every lane); the chunks in flight are kept across the
  // lanes: lane i holds chunk c with c % kRing == i (its slab count, landed barrier and the
  // barrier that frees its slabs: for a routed chunk the dequantising warps' "read", for a
  // dense one the MMAs' completion)
  uint32_t head = 0, released = 0, oldest = 0;
  uint32_t my_n = 0, my_wf = 0, my_par = 0, my_rel = 0, my_rpar = 0;
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    // claim the next work item only now that this one is needed, and publish it to the other
    // roles; entry k % kQueue is free once every reader has read its previous use
    int it = -1;
    QEntry &e = qu.slot[k % kQueue];
    if (lane == 0) {
      ok = wait_bar(qu.bars + 8 * (kIQE + k % kQueue), ((k / kQueue) & 1) ^ 1, abort_flag, a.s.err);
      // The claim counter is reset by the previous layer's combine kernel: the first claim
      // waits until that is visible, through the ready count (which the router raises only
      // after that kernel has completed) or, without shared items, the grid dependency.
      if (ok && k == 0) {
        if (n_shared > 0) {
          ok = wait_ready<PHASE>(a, abort_flag);
        } else {
          pdl_wait();
          n_items = a.s.n_items[PHASE - 1];
          routed_ready = true;
        }
      }
      if (ok) {
        it = atomicAdd(a.s.work + (PHASE - 1), 1);
        if (it < n_shared) {
          e.w = work_item(PHASE - 1, it, &n_shared, nullptr, nullptr, a.E, a.T, a.H, a.I, a.Is);
        } else {
          if (!routed_ready) {  // the previous kernels (router, gather; gate_up) have completed
            pdl_wait();
            n_items = a.s.n_items[PHASE - 1];
            routed_ready = true;
          }
          if (it >= n_items)
            it = -1;
          else
            e.w = items[it];
        }
        e.it = it;
        if (it >= 0) e.v = view_item<PHASE>(a, e.w);
        mbar_arrive(qu.bars + 8 * (kIQF + k % kQueue));
      }
    }
    __syncwarp();
    it = __shfl_sync(0xffffffffu, it, 0);
    if (it < 0) break;
    const WorkItem w = e.w;
    const ItemView v = e.v;
    // lane p < q copies plane p of every chunk; lane t < 8 copies K-step piece t of a dense tile
    const uint32_t bytes = (uint32_t)v.nr * 16;
    const uint32_t tx = v.routed ? bytes * v.q : (uint32_t)(kCtaRows * kChunkCols * 2);
    const uint8_t *src = nullptr;
    uint32_t src_step = 0, lane_slab = 0;
    if (v.routed) {
      if (lane < v.q)
        src = reinterpret_cast<const uint8_t *>(v.bd->plane[lane] + slab_word(w.tile, w.kc0, v.N, v.KC));
      src_step = bytes;  // slabs of consecutive chunks are consecutive
      lane_slab = lane;
    } else {
      src = reinterpret_cast<const uint8_t *>(v.W + ((long)w.tile * v.KC + w.kc0) * (kCtaRows * kChunkCols) +
                                              lane * 2048);
      src_step = kCtaRows * kChunkCols * 2;
      lane_slab = 2 * lane;
    }
    const bool copies = v.routed ? lane < v.q : lane < 8;
    const uint32_t cbytes = v.routed ? bytes : 2 * kSlab;
    for (int kc = w.kc0; kc < w.kc1; ++kc) {
      const uint32_t c = pos.c;
      uint32_t n, seq;
      const uint32_t base = pos.take(v.routed, v.q, S, n, seq);
      const uint32_t full = wf_bar(bars, v.routed, seq);
      // room: at most kRing chunks in flight and their slabs within the ring.  Every lane
      // checks its own chunk in flight at once, and the run of released chunks from the oldest
      // on is retired in one step; only when the oldest is still in use does lane 0 wait.
      while (head + n > released + (uint32_t)S || c - oldest >= (uint32_t)kRing) {
        const uint32_t age = ((uint32_t)lane - oldest) % kRing;  // lane < kRing holds chunk oldest + age
        const bool mine = lane < kRing && oldest + age < c;
        const bool done = mine && mbar_try_wait(my_rel, my_rpar);
        uint32_t run = (mine && !done) ? age : c - oldest;  // released chunks from the oldest on
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) run = min(run, __shfl_xor_sync(0xffffffffu, run, off));
        uint32_t freed = (mine && age < run) ? my_n : 0u;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) freed += __shfl_xor_sync(0xffffffffu, freed, off);
        released += freed;
        oldest += run;
        if (run == 0) {  // the oldest chunk is still being read: wait for it
          const uint32_t rb = __shfl_sync(0xffffffffu, my_rel, oldest % kRing);
          const uint32_t rp = __shfl_sync(0xffffffffu, my_rpar, oldest % kRing);
          if (lane == 0) ok = wait_bar(rb, rp, abort_flag, a.s.err);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          released += __shfl_sync(0xffffffffu, my_n, oldest % kRing);
          ++oldest;
        }
      }
      if (!ok) break;
      if (lane == (int)(c % kRing)) {
        my_n = n;
        my_wf = full;
        my_par = (seq / kRing) & 1;
        my_rel = bars + 8 * ((v.routed ? kRD : kWE) + seq % kRing);
        my_rpar = (seq / kRing) & 1;
      }
      head += n;
      // the copies first: a barrier's transaction count may run below zero until the expected
      // bytes are announced, and the phase cannot complete before that arrival
      if (copies) {
        if (evict_first)
          bulk_g2s_hint(ring + ring_add(base, lane_slab, S) * kSlab, src, cbytes, full, stream_policy);
        else
          bulk_g2s(ring + ring_add(base, lane_slab, S) * kSlab, src, cbytes, full);
      }
      if (lane == 0) mbar_arrive_expect_tx(full, tx);
      src += src_step;
    }
  }
  // every copy issued must land before the CTA may exit: each lane drains its chunk in flight
  __syncwarp();
  if (lane < kRing && oldest + (uint32_t)((lane - (int)(oldest % kRing) + kRing) % kRing) < pos.c)
    drain_bar(my_wf, my_par);
}

// LUT_q rows of every routed item's tile (one TMA bulk copy), as far ahead as the two slots
// allow.
template <int PHASE>
__device__ void lut_producer(const FwdArgs &a, const TcLayout &L, uint8_t *sm, uint32_t bars, const ItemQueue &qu,
                             volatile int *abort_flag) {
  if ((threadIdx.x & 31) != 0) return;
  const uint32_t lut0 = lut_base(sm, L);
  LutSched ls;
  for (uint32_t k = 0;; ++k) {
    WorkItem w;
    ItemView v;
    if (!queue_read(qu, k, 1u, abort_flag, a.s.err, w, v)) break;
    if (!v.routed) continue;
    const int q = v.q;
    bool both;
    const int slot = ls.next(q, both);
    bool ok = wait_bar(bars + 8 * (kLE + slot), (ls.uses[slot] & 1) ^ 1, abort_flag, a.s.err);
    if (ok && both) ok = wait_bar(bars + 8 * (kLE + 1), (ls.uses[1] & 1) ^ 1, abort_flag, a.s.err);
    if (!ok) break;
    ++ls.uses[slot];
    if (both) ++ls.uses[1];
    const uint32_t lbytes = (uint32_t)lut_tile_bytes(q);
    mbar_arrive_expect_tx(bars + 8 * (kLF + slot), lbytes);
    bulk_g2s(lut0 + slot * kLutSlot, v.lut + (size_t)w.tile * (lbytes / 2), lbytes, bars + 8 * (kLF + slot));
    ++ls.fills[slot];
  }
  for (int s = 0; s < 2; ++s)
    if (ls.fills[s] > 0) drain_bar(bars + 8 * (kLF + s), (ls.fills[s] - 1) & 1);
}

// The activation producer: per chunk, slot b_seq % kBSlots is refilled once the MMAs of its
// previous chunk are done; lane i loads box i (stage i / boxes, rows kBoxRows (i % boxes)
// onward) of the item's consecutive rows, all completing on the slot's barrier.
template <int PHASE, int TOK, bool GV>
__device__ void ab_producer(const FwdArgs &a, const BMaps &bm, const TcLayout &L, uint8_t *sm, uint32_t bars,
                            const ItemQueue &qu, volatile int *abort_flag) {
  using T_ = Tiling<TOK>;
  const int lane = threadIdx.x & 31;
  const uint32_t gx = smem_u32(sm) + (uint32_t)L.gx_off;
  uint32_t b_seq = 0, a_seq = 0, gx_seq[kGxSlots] = {0u, 0u, 0u, 0u};
  bool ok = true;
  // the shared expert's activations are counted ready (router rows, shared h), the routed ones
  // complete with the grid dependency; the tensor copies of every lane are ordered after what
  // lane 0 observed
  bool xh_ready = false, xs_ready = false;
  for (uint32_t k = 0; ok; ++k) {
    WorkItem w;
    ItemView v;
    if (!queue_read(qu, k, 0xffffffffu, abort_flag, a.s.err, w, v)) break;
    if (!(v.routed ? xs_ready : xh_ready)) {
      if (v.routed) {
        pdl_wait();
        xs_ready = true;
      } else {
        if (lane == 0) ok = wait_ready<PHASE>(a, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        xh_ready = true;
      }
      fence_proxy_async_global();
    }
    if (GV && v.gemv) {  // one 8-row box of 128 columns per chunk into its stream's GEMV slot
      const TmaDesc *map = PHASE == 1 ? &bm.gemv.xs : &bm.gemv.h_routed;
      for (int kc = w.kc0; kc < w.kc1; ++kc) {
        const uint32_t gs = a_seq++ % kDqStreams;
        if (lane == 0) {
          ok = wait_bar(bars + 8 * (kGXE + gs), (gx_seq[gs] & 1) ^ 1, abort_flag, a.s.err);
          if (ok) {
            mbar_arrive_expect_tx(bars + 8 * (kGXF + gs), (uint32_t)kGxBytes);
            tma_load_2d(gx + gs * kGxBytes, map, kc * kChunkCols, v.row0, bars + 8 * (kGXF + gs));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++gx_seq[gs];
      }
      continue;
    }
    if (v.routed) a_seq += (uint32_t)(w.kc1 - w.kc0);
    const ActMaps &mm = T_::kBoxRows == 16 ? bm.rows16 : bm.rows128;
    const TmaDesc *map = PHASE == 1 ? (v.routed ? &mm.xs : &mm.xh) : (v.routed ? &mm.h_routed : &mm.h_shared);
    const int rows = (v.npad + T_::kBoxRows - 1) / T_::kBoxRows * T_::kBoxRows;  // rows loaded per stage
    const int boxes = rows / T_::kBoxRows;  // per stage
    const bool loads = lane < T_::kBPieces * boxes;
    const int piece = loads ? lane / boxes : 0, rb = loads ? lane % boxes : 0;
    for (int kc = w.kc0; kc < w.kc1; ++kc) {
      const int bs = b_seq % T_::kBSlots;
      if (lane == 0) {
        ok = wait_bar(bars + 8 * (kBE + bs), ((b_seq / T_::kBSlots) & 1) ^ 1, abort_flag, a.s.err);
        if (ok) mbar_arrive_expect_tx(bars + 8 * (kBF + bs), (uint32_t)(T_::kBPieces * rows * T_::kBK * 2));
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (loads)
        tma_load_2d(b_stage<TOK>(sm, L, bs * T_::kBPieces + piece) + rb * T_::kBoxRows * T_::kBK * 2, map,
                    kc * kChunkCols + piece * T_::kBK, v.row0 + rb * T_::kBoxRows, bars + 8 * (kBF + bs));
      ++b_seq;
    }
  }
  // the last fills (the only ones whose barrier phase may still be open) land before exit
  __syncwarp();
  if (lane == 0) {
    for (uint32_t i = b_seq > (uint32_t)T_::kBSlots ? b_seq - T_::kBSlots : 0u; i < b_seq; ++i)
      drain_bar(bars + 8 * (kBF + i % T_::kBSlots), (i / T_::kBSlots) & 1);
    for (int j = 0; j < kGxSlots; ++j)
      if (gx_seq[j] > 0) drain_bar(bars + 8 * (kGXF + j), (gx_seq[j] - 1) & 1);
  }
}

// Descriptor of K-step 0 of an activation stage: 128-byte swizzled rows in 8-row atoms of
// 1 KB.  K-step t adds t kDescStep to it (the start-address field, which does not overflow
// inside shared memory).
__device__ __forceinline__ uint64_t b_desc(uint32_t stage) { return smem_desc_sw128(stage, 1024); }

// The MMA warp.  Every lane runs the loop on the same (warp-uniform) values and one elected
// lane issues the tensor-core instructions: an MMA issued this way costs about 75 cycles
// (M = 128, K = 16, any N up to 128) against about 108 from a lane that runs the loop alone,
// as its operands stay in the uniform datapath.  For a GEMV item the warp only grants the
// accumulator buffer to the dequantising warps and returns each chunk's slabs to the weight
// producer once those warps have read them.
template <int PHASE, int TOK, bool GV>
__device__ void mma_issuer(const FwdArgs &a, const TcLayout &L, uint8_t *sm, uint32_t bars, uint32_t tmem,
                           const ItemQueue &qu, volatile int *abort_flag) {
  using T_ = Tiling<TOK>;
  const uint32_t ring = smem_u32(sm) + (uint32_t)L.ring_off;
  const int S = L.slabs;
  RingPos pos;
  uint32_t a_seq = 0, item_seq = 0, m_seq = 0, gi_seq = 0;
  // next B slot and the phase parities of the B slot and A buffer barriers the next chunk waits on
  uint32_t b_slot = 0, b_par = 0, a_par = 0;
  // K-step 0 of B stage 0, and the step between stages (stages are equally spaced when they all
  // sit below the LUT slots, as in the decode tiling; the prefill tiling computes each one)
  const uint64_t bdesc0 = b_desc(b_stage<TOK>(sm, L, 0));
  const uint64_t bstep = (uint64_t)(L.b_bytes >> 4);
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    WorkItem w;
    ItemView v;
    if (!queue_read(qu, k, 0xffffffffu, abort_flag, a.s.err, w, v)) break;
    const int acs = item_seq % 2;
    ok = wait_bar_all(bars + 8 * (kAE + acs), ((item_seq / 2) & 1) ^ 1, abort_flag, a.s.err);
    if (!ok) break;
    ++item_seq;
    if (GV && v.gemv) {  // computed by the dequantising warps: grant them the accumulator buffer
      if (elect_one()) mbar_arrive(bars + 8 * (kGAG + gi_seq % 2));
      __syncwarp();
      ++gi_seq;
      for (int kc = w.kc0; kc < w.kc1 && ok; ++kc) {
        uint32_t n, seq;
        pos.take(true, v.q, S, n, seq);
        const int ts = a_seq & (T_::kAStages - 1);
        ok = wait_bar_all(bars + 8 * (kTAF + ts), a_par, abort_flag, a.s.err);
        if (((++a_seq) & (T_::kAStages - 1)) == 0) a_par ^= 1u;
        if (ok && elect_one()) tc_commit(bars + 8 * (kTAE + ts));  // after the MMAs issued so far
        __syncwarp();
      }
      continue;
    }
    const uint32_t idesc = idesc_f16_f32(128, v.npad);
    tc_fence_after();
    const uint32_t d = tmem + acs * T_::kAccCols;
    bool first = true;
    for (int kc = w.kc0; kc < w.kc1; ++kc) {
      uint32_t n, seq;
      const uint32_t base = pos.take(v.routed, v.q, S, n, seq);
      const int ts = a_seq & (T_::kAStages - 1);
      const int bs = b_slot;
      // the chunk's A operand (or dense weights) and its B slot; both checks are issued together
      ok = v.routed ? wait2_all(bars + 8 * (kTAF + ts), a_par, bars + 8 * (kBF + bs), b_par, abort_flag, a.s.err)
                    : wait2_all(wf_bar(bars, false, seq), (seq / kRing) & 1, bars + 8 * (kBF + bs), b_par, abort_flag,
                                a.s.err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc0 = first ? 0u : 1u;
      if (elect_one()) {
        if (v.routed) {
          const uint32_t at = tmem + T_::kAColBase + ts * kACols;
#pragma unroll
          for (int piece = 0; piece < T_::kBPieces; ++piece) {
            uint64_t bd;
            if constexpr (T_::kBLowStages == T_::kBStages)
              bd = bdesc0 + (uint64_t)(bs * T_::kBPieces + piece) * bstep;
            else
              bd = b_desc(b_stage<TOK>(sm, L, bs * T_::kBPieces + piece));
#pragma unroll
            for (int t = 0; t < T_::kBSteps; ++t)
              tc_mma_f16_ta(d, at + 8 * (piece * T_::kBSteps + t), bd + t * T_::kDescStep, idesc,
                            piece + t == 0 ? acc0 : 1u);
          }
          tc_commit(bars + 8 * (kBE + bs));
          tc_commit(bars + 8 * (kTAE + ts));
        } else {
#pragma unroll
          for (int piece = 0; piece < T_::kBPieces; ++piece) {
            const uint64_t bd = b_desc(b_stage<TOK>(sm, L, bs * T_::kBPieces + piece));
#pragma unroll
            for (int t = 0; t < T_::kBSteps; ++t) {
              const int kt = piece * T_::kBSteps + t;
              tc_mma_f16(d, smem_desc(ring + ring_add(base, 2 * kt, S) * kSlab, 128, 256), bd + t * T_::kDescStep,
                         idesc, kt == 0 ? acc0 : 1u);
            }
          }
          tc_commit(bars + 8 * (kBE + bs));
          tc_commit(bars + 8 * (kWE + seq % kRing));  // the dense chunk's slabs
        }
      }
      __syncwarp();
      if (++b_slot == T_::kBSlots) {
        b_slot = 0;
        b_par ^= 1u;
      }
      if (v.routed && ((++a_seq & (T_::kAStages - 1)) == 0)) a_par ^= 1u;
      first = false;
    }
    if (!ok) break;
    if (elect_one()) tc_commit(bars + 8 * (kAF + m_seq % 2));
    __syncwarp();
    ++m_seq;
  }
  // every MMA issued must complete before tensor memory is freed
  if (elect_one()) tc_commit(bars + 8 * kDrain);
  __syncwarp();
  drain_bar(bars + 8 * kDrain, 0);
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ __half2 as_h2(uint32_t u) { return *reinterpret_cast<const __half2 *>(&u); }

// Centroids of one row and one 32-column group of a routed chunk from its q plane words.
template <int Q>
__device__ __forceinline__ void dq_words(const uint32_t (&W)[8], const LutRegs &Lr, const LutLane &lu,
                                         uint32_t (&v16)[16]) {
  if constexpr (Q <= kRegLutMaxQ) {
    uint32_t S4[4];
    codes_nib<Q>(W, S4);
    dq_nib<Q>(S4, Lr, v16);
  } else {
    uint32_t Y[8];
    codes_byte<Q>(W, Y, lu.top);
    dq_byte<Q>(Y, lu, v16);
  }
}

// The dequantising warps form kDqStreams chunk streams per tensor-memory lane quarter: warp
// w serves lane quarter w & 3 and stream w >> 2, and stream j takes the routed chunks whose
// sequence number (over all routed chunks of the launch) is j modulo kDqStreams, all 128
// columns of the quarter's 32 rows.  The four warps of an SM sub-partition (which all serve
// the same lane quarter) thus work on different chunks, and their memory and barrier
// latencies do not line up.  Every barrier slot a warp waits on belongs to its own stream
// (the rings of "routed chunk landed", "slabs read" and A-buffer barriers have lengths that
// are multiples of kDqStreams, and each stream has its own GEMV activation slot), so a warp
// sees every phase of the barriers it waits on.
//
// One routed item for a dequantising warp.  The warp reads a chunk's plane words group by
// group; after the last group's words it tells the weight producer that it is done with the
// chunk's slabs (the barrier completes when the stream's four warps have), so that a routed
// chunk does not hold ring space while the tensor cores work on it.
// Tensor-core items: the four 32-column groups go to the chunk's A buffer one after the
// other, from two register sets used in turn (a set is rewritten only after the store that
// read it has completed, and that store had a group's arithmetic to complete in).  GEMV items
// (decode tiling, at most kGemvMaxTok tokens): the same centroids multiplied on the CUDA cores
// by the item's activation rows (one 8-row box of 128 columns per chunk in the stream's GEMV
// slot, read by the whole warp at one address per load), each 32-column group summed in
// packed fp16 pairs (16 products per half) and then added in fp32 to the thread's running
// dot products; at the end of the item the stream's sums go to tensor memory (columns
// 8 stream + t of the item's accumulator buffer), where the epilogue adds the streams in
// order.  Either way the warp then signals the chunk's A-buffer barrier.
template <int PHASE, int TOK, bool GV, int Q>
__device__ bool dq_item(const FwdArgs &a, const WorkItem &w, const ItemView &v, uint8_t *sm, const TcLayout &L,
                        uint32_t bars, uint32_t tmem, uint32_t lut_slot, int quarter, int stream, RingPos &pos,
                        uint32_t &a_seq, uint32_t &gx_seq, uint32_t &gi_seq, uint32_t acs, volatile int *abort_flag) {
  using T_ = Tiling<TOK>;
  const int lane = threadIdx.x & 31;
  const int r = 32 * quarter + lane;
  const bool rv = r < v.nr;
  const int S = L.slabs;
  const LutLane lu = lut_lane(lut_slot, quarter, lane);
  LutRegs Lr;
  if constexpr (Q <= kRegLutMaxQ) {
    uint32_t P[8];
    lut_pairs_smem<Q>(lu, P);
    lut_regs(P, Lr);
  }
  const uint32_t cg_off = (uint32_t)v.nr * 4;  // column-group stride inside a slab
  const uint32_t ring = smem_u32(sm) + (uint32_t)L.ring_off + (uint32_t)r * 4;
  const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
  const bool gemv = GV && TOK == kTokChunk && v.gemv;
  const uint32_t gx = smem_u32(sm) + (uint32_t)L.gx_off + (uint32_t)stream * kGxBytes;
  float acc[kGemvMaxTok];
#pragma unroll
  for (int t = 0; t < kGemvMaxTok; ++t) acc[t] = 0.f;
  uint32_t va[16], vb[16];
  for (int kc = w.kc0; kc < w.kc1; ++kc) {
    uint32_t n, seq;
    const uint32_t sl = pos.take(true, Q, S, n, seq);
    const uint32_t as = a_seq++;
    if ((int)(as % kDqStreams) != stream) continue;
    const int ts = as % T_::kAStages;
    if (!wait_bar_all(wf_bar(bars, true, seq), (seq / kRing) & 1, abort_flag, a.s.err)) return false;
    const uint32_t src = ring + sl * kSlab;
    uint32_t W[8];
    if (!gemv) {
#pragma unroll
      for (int p = 0; p < 8; ++p) W[p] = (p < Q && rv) ? lds32(src + p * kSlab) : 0u;
      dq_words<Q>(W, Lr, lu, va);
      if (!wait_bar_all(bars + 8 * (kTAE + ts), ((as / T_::kAStages) & 1) ^ 1, abort_flag, a.s.err)) return false;
      tc_fence_after();
      const uint32_t at = tmem + lane_base + T_::kAColBase + ts * kACols;
      tmem_st16(at, va);
#pragma unroll
      for (int j = 1; j < 4; ++j) {
        uint32_t(&vv)[16] = (j & 1) ? vb : va;
#pragma unroll
        for (int p = 0; p < 8; ++p) W[p] = (p < Q && rv) ? lds32(src + j * cg_off + p * kSlab) : 0u;
        if (j == 3) {
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + 8 * (kRD + seq % kRing));  // ordered after the reads
        }
        dq_words<Q>(W, Lr, lu, vv);
        tmem_wait_st();
        tmem_st16(at + 16 * j, vv);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      // (testing: a.withhold keeps back one arrival of the launch's first routed chunk, so that
      // the MMA warp's bounded wait on it expires; nothing asynchronous is held back)
      const bool keep_back = PHASE == 1 && a.withhold && as == 0 && quarter == 0;
      if (lane == 0 && !keep_back) mbar_arrive(bars + 8 * (kTAF + ts));
    } else {
      if (!wait_bar_all(bars + 8 * (kGXF + stream), gx_seq & 1, abort_flag, a.s.err)) return false;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
#pragma unroll
        for (int p = 0; p < 8; ++p) W[p] = (p < Q && rv) ? lds32(src + j * cg_off + p * kSlab) : 0u;
        if (j == 3) {
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + 8 * (kRD + seq % kRing));
        }
        dq_words<Q>(W, Lr, lu, va);
#pragma unroll
        for (int t = 0; t < kGemvMaxTok; ++t) {
          if (t < v.ntok) {
            __half2 h = __float2half2_rn(0.f);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 x4 = lds128(gx + t * (kChunkCols * 2) + 64 * j + 16 * i);
              h = __hfma2(as_h2(va[4 * i + 0]), as_h2(x4.x), h);
              h = __hfma2(as_h2(va[4 * i + 1]), as_h2(x4.y), h);
              h = __hfma2(as_h2(va[4 * i + 2]), as_h2(x4.z), h);
              h = __hfma2(as_h2(va[4 * i + 3]), as_h2(x4.w), h);
            }
            acc[t] += __low2float(h) + __high2float(h);
          }
        }
      }
      ++gx_seq;
      if (!wait_bar_all(bars + 8 * (kTAE + ts), ((as / T_::kAStages) & 1) ^ 1, abort_flag, a.s.err)) return false;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars + 8 * (kGXE + stream));
        mbar_arrive(bars + 8 * (kTAF + ts));
      }
    }
  }
  if (gemv) {  // the accumulator buffer is this item's once the MMA warp has granted it
    if (!wait_bar_all(bars + 8 * (kGAG + gi_seq % 2), (gi_seq / 2) & 1, abort_flag, a.s.err)) return false;
    tc_fence_after();
    uint32_t r8[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) r8[t] = t < kGemvMaxTok ? __float_as_uint(acc[t < kGemvMaxTok ? t : 0]) : 0u;
    tmem_st8(tmem + lane_base + acs * T_::kAccCols + 8 * stream, r8);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (kAFG + gi_seq % 2));
    ++gi_seq;
  }
  return true;
}

template <int PHASE, int TOK, bool GV>
__device__ void dequantiser(const FwdArgs &a, const TcLayout &L, uint8_t *sm, uint32_t bars, uint32_t tmem,
                            const ItemQueue &qu, volatile int *abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, stream = warp >> 2;
  const uint32_t lut0 = lut_base(sm, L);
  RingPos pos;
  uint32_t a_seq = 0, gx_seq = 0, gi_seq = 0, item_seq = 0;
  LutSched ls;
  for (uint32_t k = 0;; ++k) {
    WorkItem w;
    ItemView v;
    if (!queue_read(qu, k, 0xffffffffu, abort_flag, a.s.err, w, v)) break;
    const uint32_t acs = item_seq++ % 2;
    if (!v.routed) {  // dense chunks: only the ring position moves
      for (int kc = w.kc0; kc < w.kc1; ++kc) {
        uint32_t n, seq;
        pos.take(false, 0, L.slabs, n, seq);
      }
      continue;
    }
    bool both;
    const int slot = ls.next(v.q, both);
    if (!wait_bar_all(bars + 8 * (kLF + slot), ls.fills[slot] & 1, abort_flag, a.s.err)) return;
    ++ls.fills[slot];
    const uint32_t lut_slot = lut0 + slot * kLutSlot;
    bool ok;
    switch (v.q) {
#define PW_DQ_CASE(QQ)                                                                                          \
  case QQ:                                                                                                      \
    ok = dq_item<PHASE, TOK, GV, QQ>(a, w, v, sm, L, bars, tmem, lut_slot, quarter, stream, pos, a_seq, gx_seq, gi_seq, acs, \
                                 abort_flag);                                                                  \
    break;
      PW_DQ_CASE(1)
      PW_DQ_CASE(2)
      PW_DQ_CASE(3)
      PW_DQ_CASE(4)
      PW_DQ_CASE(5)
      PW_DQ_CASE(6)
      PW_DQ_CASE(7)
      default:
        ok = dq_item<PHASE, TOK, GV, 8>(a, w, v, sm, L, bars, tmem, lut_slot, quarter, stream, pos, a_seq, gx_seq, gi_seq, acs,
                                    abort_flag);
        break;
#undef PW_DQ_CASE
    }
    if (!ok) return;
    // the LUT slot is free once this item's last centroids are in registers
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(bars + 8 * (kLE + slot));
      if (both) mbar_arrive(bars + 8 * (kLE + 1));
    }
  }
}

template <int PHASE, int TOK, bool GV>
__device__ void epilogue(const FwdArgs &a, uint32_t bars, uint32_t tmem, const ItemQueue &qu,
                         volatile int *abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;
  uint32_t item_seq = 0, m_seq = 0, gi_seq = 0;
  for (uint32_t k = 0;; ++k) {
    WorkItem w;
    ItemView v;
    if (!queue_read(qu, k, 0xffffffffu, abort_flag, a.s.err, w, v)) break;
    const int acs = item_seq % 2;
    const bool gemv = GV && TOK == kTokChunk && v.gemv;
    bool ok;
    if (gemv) {
      ok = wait_bar_all(bars + 8 * (kAFG + gi_seq % 2), (gi_seq / 2) & 1, abort_flag, a.s.err);
      ++gi_seq;
    } else {
      ok = wait_bar_all(bars + 8 * (kAF + m_seq % 2), (m_seq / 2) & 1, abort_flag, a.s.err);
      ++m_seq;
    }
    if (!ok) return;
    tc_fence_after();
    const int row = 32 * quarter + lane;  // tile row = tensor-memory lane
    const int R = w.tile * kCtaRows + row;
    const bool empty = w.kc1 <= w.kc0;     // nothing accumulated (an empty split part)
    const uint32_t taddr = tmem + ((uint32_t)(32 * quarter) << 16) + acs * Tiling<TOK>::kAccCols;
    bool fin = true;  // every h written is a finite fp16
    for (int c = 0; c < (gemv ? 8 : v.npad); c += 8) {
      uint32_t r8[8];
      if (gemv) {  // the column-group sets' dot products, added in order
        float f8[8];
#pragma unroll
        for (int g = 0; g < kDqStreams; ++g) {
          tmem_ld8(taddr + 8 * g, r8);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) f8[i] = g == 0 ? __uint_as_float(r8[i]) : f8[i] + __uint_as_float(r8[i]);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) r8[i] = __float_as_uint(f8[i]);
      } else {
        tmem_ld8(taddr + c, r8);
        tmem_wait_ld();
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float acc = empty ? 0.f : __uint_as_float(r8[i]);
        const int j = c + i;
        if (PHASE == 1) {
          const float up = __shfl_down_sync(0xffffffffu, acc, 8);
          if ((row & 15) < 8 && R < v.N && j < v.ntok) {
            const int f = R / 16 * 8 + (R & 7);
            const float hf = silu(acc) * up;
            fin = fin && fp16_finite(hf);
            const uint16_t hv = f2h(hf);
            if (v.routed)
              a.s.h_routed[(size_t)(v.row0 + j) * a.I + f] = hv;
            else
              a.s.h_shared[(size_t)(v.row0 + j) * a.Is + f] = hv;
          }
        } else if (R < v.N && j < v.ntok) {
          if (v.routed)  // the K part's partial sums (one part but at decode batch sizes)
            a.s.o_routed[((size_t)w.part * a.T * a.K + v.row0 + j) * a.H + R] = acc;
          else
            a.s.o_shared[((size_t)w.part * a.T + v.row0 + j) * a.H + R] = acc;
        }
      }
    }
    if (PHASE == 1 && !fin) atomicOr(a.s.err, kErrRange);
    if (PHASE == 1 && !v.routed && a.s.ready) {  // this warp's rows of the shared h are written
      fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd(a.s.ready + 2 * a.layer + 1, 1);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + 8 * (kAE + acs));
    ++item_seq;
  }
}

template <int PHASE, int TOK, bool GV>
__global__ void __launch_bounds__(kTcThreads, 1) tc_ffn_kernel(FwdArgs a, TcLayout L, const __grid_constant__ BMaps bm) {
  using T_ = Tiling<TOK>;
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ int abort_flag;
  __shared__ uint32_t tmem_slot;
  __shared__ QEntry queue_slot[kQueue];
  const int warp = threadIdx.x >> 5;
  {  // regions by absolute shared address (see TcLayout)
    const uint32_t base = smem_u32(sm);
    constexpr int low = T_::kBLowStages;
    L.b_off = 0;
    L.gx_off = low * L.b_bytes;
    L.bar_off = L.gx_off + kGxSlots * kGxBytes;
    L.lut_off = (int)(kLutAddr - base);
    L.b_hi = (int)(kRingAddr - base);
    L.ring_off = L.b_hi + (T_::kBStages - low) * L.b_bytes;
    L.slabs = L.smem > L.ring_off ? ((L.smem - L.ring_off) / kSlab) & ~1 : 0;
    // a dense chunk (16 slabs, one of padding at most) must fit the ring
    const bool misaligned = ((base + L.b_off) & 1023u) != 0u;  // swizzle atoms are 1 KB-aligned
    if (base >= kLutAddr || L.bar_off + kNumBars * 8 > L.lut_off || L.slabs < kDenseSlabs + 2 || misaligned) {
      if (threadIdx.x == 0) atomicOr(a.s.err, 3);  // the map does not fit this launch
      return;
    }
  }
  const uint32_t bars = smem_u32(sm + L.bar_off);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(bars + 8 * (kRD + i), kDq / kDqStreams);  // the chunk's stream has read its slabs
      mbar_init(bars + 8 * (kWFR + i), 1);
      mbar_init(bars + 8 * (kWFD + i), 1);
      mbar_init(bars + 8 * (kWE + i), 1);
    }
    for (int i = 0; i < T_::kAStages; ++i) {
      mbar_init(bars + 8 * (kTAF + i), kDq / kDqStreams);  // the chunk's stream, one warp per lane quarter
      mbar_init(bars + 8 * (kTAE + i), 1);
    }
    for (int i = 0; i < T_::kBSlots; ++i) {
      mbar_init(bars + 8 * (kBF + i), 1);  // lane 0 of the activation producer
      mbar_init(bars + 8 * (kBE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 8 * (kLF + i), 1);
      mbar_init(bars + 8 * (kLE + i), kDq);
      mbar_init(bars + 8 * (kAF + i), 1);
      mbar_init(bars + 8 * (kAE + i), kEpi);
    }
    mbar_init(bars + 8 * kDrain, 1);
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(bars + 8 * (kIQF + i), 1);
      mbar_init(bars + 8 * (kIQE + i), kQueueReaders);
    }
    for (int i = 0; i < kGxSlots; ++i) {
      mbar_init(bars + 8 * (kGXF + i), 1);    // lane 0 of the activation producer
      mbar_init(bars + 8 * (kGXE + i), kDq / kDqStreams);  // the stream's warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bars + 8 * (kGAG + i), 1);    // the MMA warp
      mbar_init(bars + 8 * (kAFG + i), kDq);
    }
    abort_flag = 0;
    s_wait_cycles = a.wait_cycles > 0 ? a.wait_cycles : kWaitCyclesDefault;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // set up before the previous kernel of the stream has finished.  Its outputs are read per
  // role: the shared expert's items start on their counted activations, the routed items on
  // the completed grid dependency.
  pdl_trigger();
  const uint32_t tmem = tmem_slot;
  const ItemQueue qu{queue_slot, bars};
  if (warp < kDq)
    dequantiser<PHASE, TOK, GV>(a, L, sm, bars, tmem, qu, &abort_flag);
  else if (warp < kWarpP)
    epilogue<PHASE, TOK, GV>(a, bars, tmem, qu, &abort_flag);
  else if (warp == kWarpP)
    weight_producer<PHASE>(a, L, sm, bars, qu, &abort_flag);
  else if (warp == kWarpAB)
    ab_producer<PHASE, TOK, GV>(a, bm, L, sm, bars, qu, &abort_flag);
  else if (warp == kWarpMma)
    mma_issuer<PHASE, TOK, GV>(a, L, sm, bars, tmem, qu, &abort_flag);
  else
    lut_producer<PHASE>(a, L, sm, bars, qu, &abort_flag);
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int TOK, bool GV>
static int launch_tiled(const FwdArgs &a, int phase, cudaStream_t st) {
  using T_ = Tiling<TOK>;
  TcLayout L{};
  L.npad_max = TOK;
  L.b_bytes = L.npad_max * T_::kBK * 2;
  if (!a.bmaps) return (int)cudaErrorInvalidValue;
  const BMaps bm = *a.bmaps;
  L.smem = kSmemLimit;
  if (T_::kBLowStages * L.b_bytes + kGxSlots * kGxBytes + kNumBars * 8 + 2048 > (int)kLutAddr)
    return (int)cudaErrorInvalidConfiguration;
  const int max_items = phase == 1 ? a.s.max_items1 : a.s.max_items2;
  const int grid = min(max_items, a.sm_count);
  if (phase == 1) {
    cudaFuncSetAttribute(tc_ffn_kernel<1, TOK, GV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
    return (int)launch_pdl(tc_ffn_kernel<1, TOK, GV>, dim3(grid), dim3(kTcThreads), (size_t)L.smem, st, a, L, bm);
  }
  cudaFuncSetAttribute(tc_ffn_kernel<2, TOK, GV>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
  return (int)launch_pdl(tc_ffn_kernel<2, TOK, GV>, dim3(grid), dim3(kTcThreads), (size_t)L.smem, st, a, L, bm);
}

// The kernel image with the GEMV items' code is launched only when some item may take that
// path; the tensor-core-only image is smaller, which keeps instruction fetch out of the way.
int launch_ffn(const FwdArgs &a, int phase, void *stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (tok_chunk_for(a.T) == kTokChunkPrefill) return launch_tiled<kTokChunkPrefill, false>(a, phase, st);
  return a.gemv_max > 0 ? launch_tiled<kTokChunk, true>(a, phase, st) : launch_tiled<kTokChunk, false>(a, phase, st);
}

}  // namespace pw
