// pw_internal.h -- structures and index maps shared by the host runtime and the kernels.
//
// Kernel-private plane tiling (the ABI layout is restored by pw_unpack_indices):
//   A block's device rows are grouped in CTA tiles of 128 rows (the last may hold fewer; N is
//   a multiple of 16).  For a gate_up block each 16-row group holds 8 gate rows followed by
//   the 8 up rows of the same 8 features, so that gate and up of a feature sit 8 tensor-
//   memory lanes apart.  Columns are grouped in chunks of 128 (the plane row is zero-padded
//   to a multiple of 128 bits) and each chunk in 4 column groups of 32.
//   One plane of one (CTA tile, chunk) is a contiguous slab of nr x 4 words (nr = rows of
//   the tile), ordered [column group][row]; slabs are ordered [tile][chunk].  Inside a word,
//   bit (4 i + j) holds column 8 j + i of the 32-column group (i = 0..7, j = 0..3): a 4x4
//   bit transpose across the planes of a row then yields 4-bit codes of 8 consecutive
//   columns per word, and an 8x8 transpose yields 8-bit codes of 4 columns per word.
#pragma once
#include <math.h>
#include <stdint.h>

#ifdef __CUDACC__
#define PW_HD __host__ __device__ __forceinline__
#else
#define PW_HD inline
#endif

namespace pw {

constexpr int kMaxPlanes = 8;
constexpr int kChunkCols = 128;   // columns per plane chunk (one pipeline stage)
constexpr int kCtaRows = 128;     // rows per CTA tile (tensor-memory lanes of one MMA)
constexpr int kTokChunk = 64;     // tokens per work item at decode batch sizes
constexpr int kTokChunkPrefill = 128;  // tokens per work item for prefill-sized batches
constexpr int kPrefillMinT = 512;      // batches of at least this many tokens use the prefill tiling

// Tokens per work item for a launch of T tokens: the prefill tiling halves how often each
// weight tile is dequantised when experts see hundreds of tokens.
PW_HD int tok_chunk_for(int T) { return T >= kPrefillMinT ? kTokChunkPrefill : kTokChunk; }

constexpr int kRtTok = 8;  // tokens per router CTA (one warp each in top-K)
constexpr int kRtExp = 8;  // experts per router CTA (one warp each for the logits)
// CTAs of a router launch: (token groups) x (expert groups).
PW_HD int route_ctas(int T, int E) { return ((T + kRtTok - 1) / kRtTok) * ((E + kRtExp - 1) / kRtExp); }

// One row of the device weight page table (PagedWeight Sec. 3.1).  The kernels read q and
// the pointers of the block they run; commits rewrite the whole row between launches.
struct BlockDev {
  const uint32_t *plane[kMaxPlanes];  // tiled bit-planes (poison page when not resident)
  const uint16_t *lut[9];             // LUT_b in device row order (poison page when absent)
  int q;                              // committed bitwidth
  int N, K, KC;                       // rows, columns, 128-column chunks
};

// A unit of work of the expert kernels.
struct WorkItem {
  int kind;    // 0 routed expert, 1 shared expert
  int expert;  // routed expert id (kind 0)
  int tile;    // CTA row tile (kCtaRows rows)
  int tok0;    // first slot (routed: into the expert-sorted pair list; shared: token)
  int ntok;    // tokens in this item (<= tok_chunk_for(T))
  int kc0, kc1;  // 128-column stages [kc0, kc1) of the item along K
  int part;    // shared down projection: the partial-sum buffer this item writes
};

PW_HD int kpad_cols(int K) { return (K + kChunkCols - 1) / kChunkCols * kChunkCols; }

// The shared expert's down projection (K = Is) is split along K into this many items per
// row tile, so that each is about as long as a routed down item (K = I); the parts are
// summed, in order, by the combine kernel.
// Every part holds at least one stage: parts are ceil(stages / n) stages long, so when the
// cap of 8 applies the count is what that length needs (9 stages in parts of 2 make 5).
PW_HD int shared_down_splits(int I, int Is) {
  if (Is <= 0) return 1;
  const int sh = (Is / 16 + 7) / 8;           // 128-column stages of the shared down
  const int rt = kpad_cols(I) / kChunkCols;   // stages of a routed down
  int n = (sh + rt - 1) / rt;
  n = n < 1 ? 1 : (n > 8 ? 8 : n);
  const int per = (sh + n - 1) / n;
  return (sh + per - 1) / per;
}

// The routed down projection (K = I) is split along K into this many parts per (row tile,
// slot chunk) at decode batch sizes, so that a launch of a few long items (8 experts of
// 112 stages, say) becomes many of about 16 stages; each part writes its own partial-sum
// buffer, which the combine kernel adds in order.  Prefill-sized batches have items enough
// and keep one part.  Every part holds at least one stage.
PW_HD int routed_down_splits(int T, int I) {
  const int st = kpad_cols(I) / kChunkCols;
  if (T >= kPrefillMinT || st <= 16) return 1;
  int n = (st + 15) / 16;
  n = n < 1 ? 1 : (n > 8 ? 8 : n);
  const int per = (st + n - 1) / n;
  return (st + per - 1) / per;
}

// Work-list tables of one launch, written by the router's last CTA: for each projection u
// (0 gate_up, 1 down) first[u][r] = the first work item of the expert at rank r (ranks by
// decreasing committed bitwidth, ties by expert id; first[u][0] = the shared expert's item
// count, first[u][E] = the total) and rk[u][r] = that expert.  Row stride kRankStride.
constexpr int kRankStride = 257;

// Work item i of projection u from the tables and the expert-sorted slot offsets off[0..E].
// Items [0, first[0]) are the shared expert's: (row tile, token chunk), and for the down
// projection also the K part, with the chunks and parts of a tile consecutive.  Items
// [first[r], first[r + 1]) are the expert at rank r's: (row tile, slot chunk) with the slot
// chunks of a row tile consecutive, so that CTAs claiming them together share the tile's
// planes in L2; for the down projection each (row tile, K part) has its slot chunks
// consecutive, the parts of a tile one after the other.
// Number of the shared expert's work items of projection u (they lead both lists).
PW_HD int shared_item_count(int u, int T, int H, int I, int Is) {
  if (Is <= 0) return 0;
  const int tc = tok_chunk_for(T), tchunks = (T + tc - 1) / tc;
  return u == 0 ? ((2 * Is + kCtaRows - 1) / kCtaRows) * tchunks
                : ((H + kCtaRows - 1) / kCtaRows) * tchunks * shared_down_splits(I, Is);
}

PW_HD WorkItem work_item(int u, int i, const int *first, const int *rk, const int *off, int E, int T, int H,
                         int I, int Is) {
  const int tc = tok_chunk_for(T), tchunks = (T + tc - 1) / tc;
  const int kc_gu = kpad_cols(H) / kChunkCols, kc_d = kpad_cols(I) / kChunkCols;
  WorkItem w;
  if (i < first[0]) {
    int tile, c, kc0 = 0, kc1 = kc_gu, part = 0;
    if (u == 0) {
      tile = i / tchunks;
      c = i - tile * tchunks;
    } else {
      const int nsplit = shared_down_splits(I, Is);
      const int total = (Is / 16 + 7) / 8, per = (total + nsplit - 1) / nsplit;
      tile = i / (tchunks * nsplit);
      const int rem = i - tile * tchunks * nsplit;
      c = rem / nsplit;
      part = rem - c * nsplit;
      kc0 = part * per;
      kc1 = total < (part + 1) * per ? total : (part + 1) * per;
    }
    w.kind = 1;
    w.expert = 0;
    w.tile = tile;
    w.tok0 = c * tc;
    w.ntok = tc < T - c * tc ? tc : T - c * tc;
    w.kc0 = kc0;
    w.kc1 = kc1;
    w.part = part;
    return w;
  }
  int lo = 0, hi = E - 1;  // the largest rank r with first[r] <= i
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (first[mid] <= i)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int e = rk[lo], cnt = off[e + 1] - off[e], ch = (cnt + tc - 1) / tc, loc = i - first[lo];
  const int np = u ? routed_down_splits(T, I) : 1;  // K parts
  const int kcn = u ? kc_d : kc_gu;
  w.kind = 0;
  w.expert = e;
  if (np == 1) {  // the whole K (every gate_up, and every down but long ones at decode sizes)
    const int tile = loc / ch, c = loc - tile * ch;
    w.tile = tile;
    w.tok0 = c * tc;
    w.ntok = tc < cnt - c * tc ? tc : cnt - c * tc;
    w.kc0 = 0;
    w.kc1 = kcn;
    w.part = 0;
    return w;
  }
  const int tile = loc / (np * ch), rem = loc - tile * np * ch;
  const int part = rem / ch, c = rem - part * ch;
  const int per = (kcn + np - 1) / np;
  w.tile = tile;
  w.tok0 = c * tc;
  w.ntok = tc < cnt - c * tc ? tc : cnt - c * tc;
  w.kc0 = part * per;
  w.kc1 = kcn < (part + 1) * per ? kcn : (part + 1) * per;
  w.part = part;
  return w;
}

// device row of an original row (u = 0 gate_up with I features, u = 1 identity)
PW_HD int dev_row(int r, int u, int I) {
  if (u != 0) return r;
  int half = r >= I ? 1 : 0;
  int f = half ? r - I : r;
  return (f / 8) * 16 + half * 8 + (f % 8);
}
PW_HD int orig_row(int d, int u, int I) {
  if (u != 0) return d;
  int rt = d / 16, ri = d % 16;
  int f = rt * 8 + (ri % 8);
  return (ri >= 8) ? I + f : f;
}

// rows of CTA tile ct of a block with N rows
PW_HD int tile_rows(int ct, int N) { return N - ct * kCtaRows < kCtaRows ? N - ct * kCtaRows : kCtaRows; }

// first word of the slab of (CTA tile ct, chunk kc) inside a tiled plane; nr x 4 words follow
PW_HD long slab_word(int ct, int kc, int N, int KC) {
  return ((long)ct * kCtaRows * KC + (long)kc * tile_rows(ct, N)) * 4;
}

// word index inside a tiled plane and bit inside that word for (device row d, column k)
PW_HD void tile_pos(int d, int k, int N, int KC, long *word, int *bit) {
  const int ct = d / kCtaRows, r = d % kCtaRows;
  const int kc = k / kChunkCols, kk = k % kChunkCols;
  const int cg = kk / 32, j = (kk % 32) / 8, i = kk % 8;
  *word = slab_word(ct, kc, N, KC) + (long)cg * tile_rows(ct, N) + r;
  *bit = 4 * i + j;
}

// Kernel-private LUT layout of one bitwidth b of a block: per 128-row tile (the last tile
// zero-padded to 128 rows), 2^b codes of 256 bytes each; inside a code's 256 bytes, 32-bit
// word (qp * 32 + L) (qp = 0, 1; L = 0..31) holds in its low half the centroid of row
// 64 qp + L and in its high half that of row 64 qp + 32 + L.  A warp that owns the 32 rows
// 32 m + L (a tensor-memory lane quarter m) thus reads one word per lane, every lane in its
// own bank, and the code of an entry is byte 1 of its address relative to a 64 KB-aligned
// table base.
PW_HD long lut_tile_bytes(int b) { return 256L << b; }
PW_HD long lut_dev_bytes(int N, int b) { return (long)((N + kCtaRows - 1) / kCtaRows) * lut_tile_bytes(b); }
// element index (uint16) of (device row d, code c) in that layout
PW_HD long lut_dev_index(int d, int c, int b) {
  const int ct = d / kCtaRows, r = d % kCtaRows;
  const int m = r / 32, L = r % 32;
  return ct * (lut_tile_bytes(b) / 2) + ((long)c * 64 + (m >> 1) * 32 + L) * 2 + (m & 1);
}

// Kernel-private layout of dense fp16 shared-expert weights (N x K): rows padded to a
// multiple of 128, columns to a multiple of 128.  Each (128-row tile, 128-column chunk) is a
// contiguous 32 KB operand tile, tiles ordered [tile][chunk]; inside it, the eight 16-column
// K-steps of one MMA each are contiguous 4 KB pieces, and a piece holds the 16 row groups of
// 8 rows, each as two 8x8 core matrices (columns 0..7, 8..15 of the step) of 128 bytes.
// One piece is thus one MMA's A operand with a 128-byte K stride and a 256-byte row-group
// stride, and the pieces of a tile may sit anywhere in shared memory.
PW_HD long shared_tile_index(int d, int k, int K) {
  const int KCh = kpad_cols(K) / kChunkCols;
  const int r = d % kCtaRows, c = k % kChunkCols;
  return ((long)(d / kCtaRows) * KCh + k / kChunkCols) * (kCtaRows * kChunkCols) + (c / 16) * 2048 +
         (r / 8) * 128 + ((c % 16) / 8) * 64 + (r % 8) * 8 + (c % 8);
}

}  // namespace pw

// ------------------------------------------------------------------ kernel launchers
// Implemented in the .cu files; called by the host runtime.  Each returns a cudaError_t
// value as int.
namespace pw {

// An encoded TMA tensor descriptor (the driver's 128-byte, 64-byte-aligned CUtensorMap),
// opaque here; the host runtime encodes it.
struct alignas(64) TmaDesc {
  unsigned char bytes[128];
};

// Tensor maps of the expert kernels' activation tiles: fp16, boxes of 64 columns by 16 rows
// (decode tiling: as many boxes as an item has tokens) or by 128 rows (prefill tiling: one
// box per stage), 128-byte swizzle (the K-major operand layout the MMAs read), rows past the
// end read as zeros.  Rows are the scratch buffers' full capacity (max_tokens), so the maps
// are fixed for the context.
struct ActMaps {
  TmaDesc xs;        // [Tm*K][H] layer input gathered into expert-sorted slot order (routed gate_up)
  TmaDesc xh;        // [Tm][H] layer input (shared gate_up)
  TmaDesc h_routed;  // [Tm*K][I] (routed down)
  TmaDesc h_shared;  // [Tm][Is] (shared down)
};
// Activation rows of the CUDA-core (GEMV) work items: boxes of 128 columns by 8 rows, no
// swizzle (row t of a box at byte 256 t), rows past the end read as zeros.
struct GemvMaps {
  TmaDesc xs;        // [Tm*K][H] routed gate_up input in slot order
  TmaDesc h_routed;  // [Tm*K][I] routed down input
};
struct BMaps {
  ActMaps rows16, rows128;
  GemvMaps gemv;
};

struct Scratch {
  float *logits;       // [Tm][E]
  int *ids;            // [Tm][K]
  float *w;            // [Tm][K]
  int *ranks;          // [4][kRankStride] work-list tables: first[2][E + 1], then rk[2][E]
  int *offsets;        // [E + 1]
  int *slot_tok;       // [Tm*K] token of each expert-sorted slot
  int *pair_slot;      // [Tm*K] slot of pair (t, k)
  float *slot_w;       // [Tm*K] routing weight of each slot
  WorkItem *items1;    // gate_up work
  WorkItem *items2;    // down work
  int *n_items;        // [2]
  unsigned *ticket;    // [1 + ceil(Tm/8)] router last-CTA counters: all token groups, then per group
  int *ready;          // [L][2] per layer: [0] router CTAs that have written its fp16 input rows
                       // (the gate_up kernel starts the shared expert's items once all have),
                       // [1] gate_up epilogue warps done with a shared item (the down kernel
                       // starts the shared expert's items once all are); reset with the claim
                       // counters by the layer's combine kernel.  NULL: not counted
  uint16_t *xh;        // fp16 [Tm][H]: the layer input as the experts read it (normalised under PW_PRENORM)
  uint16_t *xs;        // fp16 [Tm*K][H]: xh rows in expert-sorted slot order
  uint16_t *h_routed;  // fp16 [Tm*K][I]
  uint16_t *h_shared;  // fp16 [Tm][Is]
  float *o_routed;     // [parts][T*K][H] partial sums of the routed down projection (routed_down_splits)
  float *o_shared;     // [splits][T][H] partial sums of the shared down projection
  float *inv_rms;      // [Tm] per-token 1/rms of the layer input (PW_PRENORM)
  float *sgate;        // [Tm] per-token shared-expert gate sigmoid(x . w_sg) (layers with a gate)
  float *xnorm;        // [Tm] per-token L2 norm of the layer input as the experts read it
  double *stat_count;  // [L][E]
  double *stat_wsum;   // [L][E]
  double *stat_phi;    // [L][E][4] routed-input sums for Eq. 5: sum r, sum r n, sum r n^2, max n
  int *err;            // [1] error bits: kErrWaitMask = a bounded wait gave up (1 expert kernel,
                       // 2 router, 3 tensor map), kErrRange = an fp16 activation or y not finite
  int *work;           // [2] next unclaimed work item of the two expert kernels (reset by the router)
  int max_items1, max_items2;
};

struct LayerDev {
  const float *Wr;         // [E][H]
  const float *bias;       // [E] or null
  const uint16_t *wgu;     // shared gate_up, fp16, frag16 layout (dev rows interleaved)
  const uint16_t *wd;      // shared down, fp16, frag16 layout
  const float *wsg;        // [H] shared-expert gate, or null (ungated)
};

struct FwdArgs {
  int layer, T, E, H, I, K, Is, renorm, flags;
  int stat_layer;         // row of the routing statistics the router adds to (the layer, or 0 for discarded slots)
  const BlockDev *table;  // device page table
  LayerDev lay;
  Scratch s;
  const uint16_t *x;      // bf16 [T][H]
  uint16_t *y;            // bf16 [T][H]
  int *ids_out;           // optional
  float *w_out;           // optional
  int sm_count;
  int gemv_max;           // routed work items of at most this many tokens run on the CUDA cores (decode tiling)
  long long wait_cycles;  // a bounded device wait of the expert kernels gives up after this many SM cycles
  int withhold;           // testing: 1 = the gate_up kernel withholds one A-buffer arrival (its wait expires)
  const BMaps *bmaps;     // host copy of the activation tensor maps
};
constexpr int kGemvMaxTokens = 8;      // largest GEMV item
constexpr long long kWaitCyclesDefault = 1LL << 32;  // bounded device waits: about 2 s of SM clock
constexpr int kErrWaitMask = 0xFF;  // error-word bits of the bounded waits
constexpr int kErrRange = 0x100;    // an fp16 activation (x or h) overflowed, or y is not finite
// |v| < 65520 rounds to a finite fp16 (65504 at most); NaN fails the test too.
PW_HD bool fp16_finite(float v) { return fabsf(v) < 65520.f; }
constexpr int kGemvDefaultTokens = 0;  // default threshold of a context (the tensor cores measured faster)

// ev: null, or five timing events recorded before, between and after the four kernels
int launch_forward(const FwdArgs &a, void *stream, void *const *ev);
int launch_ffn(const FwdArgs &a, int phase, void *stream);
int launch_commit(BlockDev *table, int block, const BlockDev &val, void *stream);
int launch_pack(const uint8_t *idx, int N, int K, int KC, int u, int I, int bmax,
                uint32_t *const *plane_out, void *stream);
int launch_lut_permute(const uint16_t *lut_in, int N, int entries, int u, int I,
                       uint16_t *lut_out, void *stream);
int launch_frag16(const uint16_t *w_in, int N, int K, int u, int I, uint16_t *w_out, int *bad,
                  void *stream);
int launch_unpack(const BlockDev *table, int block, int b, int u, int I, int N, int KC,
                  uint8_t *idx_out, uint16_t *w_out, void *stream);

}  // namespace pw

// ------------------------------------------------------------------ routing-only launches
#include "../../include/pw.h"
namespace pw {
int launch_route(const FwdArgs &a, void *stream);
pw_status route_args(pw_ctx *c, int layer, const void *x, int T, int32_t *ids, float *w, int flags,
                     FwdArgs *a);
pw_status report(pw_ctx *c, pw_status st, const char *msg);
int ctx_device(const pw_ctx *c);
}  // namespace pw
