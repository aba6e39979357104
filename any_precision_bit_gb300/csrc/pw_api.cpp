// pw_api.cpp -- host runtime behind include/pw.h: context, weight page table, page pools,
// packing, forward dispatch (with CUDA-graph replay of the layer stack) and the
// asynchronous offload / reload protocol of PagedWeight Sec. 3.1 and Sec. 3.3.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "../../include/pw.h"
#include "pw_internal.h"

using namespace pw;

namespace {

thread_local std::string g_thread_err;

// 2-D fp16 tensor map over a row-major [rows][cols] buffer: boxes of 64 columns (128 bytes)
// by box_rows rows with the 128-byte swizzle (or, with box_cols = 128, 128 columns by box_rows
// rows without swizzle), out-of-range elements read as zero.  The encoder is the driver's,
// looked up through the runtime (no link-time dependency on the driver library).
bool encode_act_map(TmaDesc *out, void *base, long rows, long cols, unsigned box_rows, unsigned box_cols = 64) {
  using Encode = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Encode fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
      cudaGetLastError();
      return false;
    }
    fn = reinterpret_cast<Encode>(p);
  }
  static_assert(sizeof(CUtensorMap) == sizeof(TmaDesc), "tensor map size");
  const cuuint64_t dim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t stride[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return fn(reinterpret_cast<CUtensorMap *>(out), CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dim, stride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ page pools
// Size-class free lists over large reservations.  Pages of one block type all have the
// same size, so a retired page is reused as-is by the next page of that size.
struct Pool {
  bool pinned = false;
  size_t chunk = size_t(256) << 20;
  std::vector<void *> chunks;
  std::vector<size_t> chunk_sizes;
  char *cur = nullptr;
  size_t cur_left = 0;
  std::map<size_t, std::vector<void *>> free_lists;
  int64_t reserved = 0;
  int64_t free_bytes = 0;

  static size_t round(size_t n) { return (n + 255) & ~size_t(255); }

  void *alloc(size_t n) {
    n = round(n);
    auto it = free_lists.find(n);
    if (it != free_lists.end() && !it->second.empty()) {
      void *p = it->second.back();
      it->second.pop_back();
      free_bytes -= (int64_t)n;
      return p;
    }
    if (cur_left < n) {
      size_t sz = std::max(chunk, n);
      void *p = nullptr;
      cudaError_t e = pinned ? cudaHostAlloc(&p, sz, cudaHostAllocDefault) : cudaMalloc(&p, sz);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
      }
      chunks.push_back(p);
      chunk_sizes.push_back(sz);
      reserved += (int64_t)sz;
      if (cur_left) free_bytes += (int64_t)cur_left;  // the tail of the old chunk is lost
      cur = static_cast<char *>(p);
      cur_left = sz;
    }
    void *p = cur;
    cur += n;
    cur_left -= n;
    return p;
  }
  void release(void *p, size_t n) {
    if (!p) return;
    n = round(n);
    free_lists[n].push_back(p);
    free_bytes += (int64_t)n;
  }
  void destroy() {
    for (void *p : chunks) {
      if (pinned)
        cudaFreeHost(p);
      else
        cudaFree(p);
    }
    chunks.clear();
  }
};

struct Pending {
  int kind = 0;  // 0 none, 1 offload, 2 reload
  int from = 0, to = 0;
  bool failed = false;
  unsigned new_luts = 0;  // reload: LUT pages allocated by this transfer (bit b)
};

struct HostBlock {
  bool packed = false;
  int layer = 0, expert = 0, u = 0, N = 0, K = 0, KC = 0;
  int q = 0, d = 0, q_init = 0;
  size_t plane_bytes = 0;
  size_t lut_bytes[9] = {};
  void *dplane[kMaxPlanes] = {};
  void *dlut[9] = {};
  void *hplane[kMaxPlanes] = {};
  void *hlut[9] = {};
  int state[kMaxPlanes] = {};
  Pending pend;
  bool landed = false;  // a reload's copies have landed; the raise waits for pw_commit
  int io_error = 0;     // 1 failed offload copy, 2 failed reload copy (reported by pw_commit)
  cudaEvent_t ev = nullptr;
};

struct GraphEntry {
  void *x;
  int T;
  int profiling;
  cudaStream_t stream;
  cudaGraphExec_t exec;
};

}  // namespace

struct pw_ctx {
  pw_desc d{};
  int n_bits = 0;
  int bits[9] = {};
  int sm_count = 0;
  cudaStream_t compute = nullptr, io = nullptr;
  cudaStream_t own_compute = nullptr;  // created by the context (destroyed with it)
  int profiling = 0;
  std::vector<cudaEvent_t> prof_ev;  // [L][5] timing events around the four kernels
  BlockDev *table = nullptr;
  std::vector<HostBlock> blocks;
  std::vector<LayerDev> layers;
  std::vector<int> router_set, shared_set, packed_count;
  Pool dpool, hpool;
  void *poison = nullptr;
  size_t poison_bytes = 0;
  Scratch s{};
  std::vector<void *> scratch_allocs;
  int64_t scratch_bytes = 0;
  void *stage = nullptr;  // device staging for packing / inspection
  size_t stage_bytes = 0;
  void *xdev = nullptr;   // device activations of pw_stack_forward_host
  BMaps bmaps{};          // activation tensor maps of the expert kernels (valid when has_bmaps)
  bool has_bmaps = false;
  std::vector<GraphEntry> graphs;
  std::string err;
  int sticky = 0;
  int fault_copy = 0, fault_alloc = 0;
  int hold = 0;  // testing: transfers are not observed as landed while set
  int gemv_max = kGemvDefaultTokens;  // routed items of at most this many tokens run on the CUDA cores
  int fault_withhold = 0;              // testing: the next forward withholds one device barrier arrival
  long long wait_cycles = kWaitCyclesDefault;  // bounded device waits of the expert kernels
};

namespace {

pw_status fail(pw_ctx *c, pw_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c)
    c->err = buf;
  else
    g_thread_err = buf;
  return st;
}

#define CU(c, call)                                                                   \
  do {                                                                                \
    cudaError_t _e = (call);                                                          \
    if (_e != cudaSuccess) {                                                          \
      cudaGetLastError();                                                             \
      return fail((c), PW_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(_e)); \
    }                                                                                 \
  } while (0)

bool supported(const pw_ctx *c, int b) { return b >= 1 && b <= 8 && ((c->d.bits_mask >> b) & 1u); }

void block_shape(const pw_ctx *c, int u, int *N, int *K) {
  if (u == 0) {
    *N = 2 * c->d.I;
    *K = c->d.H;
  } else {
    *N = c->d.H;
    *K = c->d.I;
  }
}

int64_t block_M(const pw_ctx *c, const HostBlock &b, int q) {
  int64_t m = (int64_t)q * (int64_t)b.plane_bytes;
  for (int i = 0; i < c->n_bits; ++i)
    if (c->bits[i] <= q) m += (int64_t)b.N * (1 << c->bits[i]) * 2;
  return m;
}

BlockDev dev_entry(const pw_ctx *c, const HostBlock &b, int q) {
  BlockDev v{};
  for (int p = 0; p < kMaxPlanes; ++p)
    v.plane[p] = static_cast<const uint32_t *>((p < q && b.dplane[p]) ? b.dplane[p] : c->poison);
  for (int bb = 0; bb <= 8; ++bb)
    v.lut[bb] = static_cast<const uint16_t *>((bb <= q && b.dlut[bb]) ? b.dlut[bb] : c->poison);
  v.q = q;
  v.N = b.N;
  v.K = b.K;
  v.KC = b.KC;
  return v;
}

pw_status check_sticky(pw_ctx *c) {
  if (c->sticky) return fail(c, PW_ERR_CUDA, "an earlier asynchronous CUDA error is sticky on this context");
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    c->sticky = 1;
    return fail(c, PW_ERR_CUDA, "asynchronous CUDA error: %s", cudaGetErrorString(e));
  }
  return PW_OK;
}

pw_status ensure_stage(pw_ctx *c, size_t n) {
  if (c->stage_bytes >= n) return PW_OK;
  if (c->stage) cudaFree(c->stage);
  c->stage = nullptr;
  c->stage_bytes = 0;
  CU(c, cudaMalloc(&c->stage, n));
  c->stage_bytes = n;
  return PW_OK;
}

bool is_device_ptr(const void *p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

void *dev_alloc_page(pw_ctx *c, size_t n) {
  if (c->fault_alloc > 0 && --c->fault_alloc == 0) return nullptr;
  return c->dpool.alloc(n);
}

pw_status observe(pw_ctx *c, int id);

void drop_graphs(pw_ctx *c) {
  for (auto &g : c->graphs) cudaGraphExecDestroy(g.exec);
  c->graphs.clear();
}

}  // namespace

// ================================================================== lifetime
extern "C" {

const char *pw_version(void) { return "pagedweight-gb300 0.1 (sm_103a)"; }

const char *pw_last_error(const pw_ctx *ctx) { return ctx ? ctx->err.c_str() : g_thread_err.c_str(); }

pw_status pw_create(const pw_desc *desc, pw_ctx **out) {
  if (!desc || !out) return fail(nullptr, PW_ERR_INVALID, "null argument");
  *out = nullptr;
  const pw_desc &d = *desc;
  if (d.L < 1 || d.E < 1 || d.E > 256 || d.K < 1 || d.K > 8 || d.K > d.E)
    return fail(nullptr, PW_ERR_INVALID, "need 1 <= K <= 8, K <= E <= 256, L >= 1");
  if (d.H < 16 || d.H % 16 || d.H > 8192) return fail(nullptr, PW_ERR_INVALID, "H must be a multiple of 16 in [16, 8192]");
  if (d.I < 8 || d.I % 8) return fail(nullptr, PW_ERR_INVALID, "I must be a positive multiple of 8");
  if (d.Is < 0 || d.Is % 16) return fail(nullptr, PW_ERR_INVALID, "Is must be a multiple of 16 (0 = none)");
  if (d.bmax < 1 || d.bmax > 8) return fail(nullptr, PW_ERR_INVALID, "bmax must be in 1..8");
  if (d.max_tokens < 1 || d.max_tokens > 65536) return fail(nullptr, PW_ERR_INVALID, "max_tokens must be in 1..65536");
  if ((d.bits_mask & ~(((1u << (d.bmax + 1)) - 1u) & ~1u)) || d.bits_mask == 0)
    return fail(nullptr, PW_ERR_INVALID, "bits_mask must name bitwidths within 1..bmax");

  pw_ctx *c = new pw_ctx();
  c->d = d;
  for (int b = 1; b <= 8; ++b)
    if ((d.bits_mask >> b) & 1u) c->bits[c->n_bits++] = b;
  c->hpool.pinned = true;
  c->hpool.chunk = size_t(64) << 20;
  auto bail = [&](pw_status st) {
    pw_destroy(c);
    return st;
  };
  if (cudaSetDevice(d.device) != cudaSuccess) {
    cudaGetLastError();
    fail(nullptr, PW_ERR_CUDA, "cudaSetDevice(%d) failed", d.device);
    delete c;
    return PW_ERR_CUDA;
  }
  cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, d.device);
  if (cudaStreamCreateWithFlags(&c->own_compute, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&c->io, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    fail(nullptr, PW_ERR_CUDA, "stream creation failed");
    return bail(PW_ERR_CUDA);
  }
  c->compute = c->own_compute;
  const int nblk = d.L * d.E * 2;
  c->blocks.resize(nblk);
  c->layers.assign(d.L, LayerDev{});
  c->router_set.assign(d.L, 0);
  c->shared_set.assign(d.L, 0);
  c->packed_count.assign(d.L, 0);
  for (int i = 0; i < nblk; ++i) {
    HostBlock &b = c->blocks[i];
    b.u = i % 2;
    b.expert = (i / 2) % d.E;
    b.layer = i / 2 / d.E;
    block_shape(c, b.u, &b.N, &b.K);
    b.KC = kpad_cols(b.K) / kChunkCols;
    b.plane_bytes = (size_t)b.N * kpad_cols(b.K) / 8;
    for (int bb = 1; bb <= 8; ++bb) b.lut_bytes[bb] = (size_t)lut_dev_bytes(b.N, bb);  // device layout
    for (int p = 0; p < kMaxPlanes; ++p) b.state[p] = PW_PAGE_CPU;
    if (cudaEventCreateWithFlags(&b.ev, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      fail(nullptr, PW_ERR_CUDA, "event creation failed");
      return bail(PW_ERR_CUDA);
    }
  }
  // poison page: large enough for any plane or LUT a kernel might touch
  size_t pmax = 0;
  for (int u = 0; u < 2; ++u) {
    int N, K;
    block_shape(c, u, &N, &K);
    pmax = std::max(pmax, (size_t)N * kpad_cols(K) / 8);
    pmax = std::max(pmax, (size_t)lut_dev_bytes(N, 8));
  }
  c->poison_bytes = pmax;
  if (cudaMalloc(&c->poison, pmax) != cudaSuccess || cudaMemset(c->poison, 0xFF, pmax) != cudaSuccess) {
    cudaGetLastError();
    fail(nullptr, PW_ERR_OOM, "poison page allocation failed");
    return bail(PW_ERR_OOM);
  }
  if (cudaMalloc(&c->table, sizeof(BlockDev) * nblk) != cudaSuccess) {
    cudaGetLastError();
    fail(nullptr, PW_ERR_OOM, "page table allocation failed");
    return bail(PW_ERR_OOM);
  }
  {
    std::vector<BlockDev> init(nblk);
    for (int i = 0; i < nblk; ++i) init[i] = dev_entry(c, c->blocks[i], 0);
    cudaMemcpy(c->table, init.data(), sizeof(BlockDev) * nblk, cudaMemcpyHostToDevice);
  }
  // forward scratch
  const long Tm = d.max_tokens, TK = Tm * d.K;
  const int tiles1 = (2 * d.I + kCtaRows - 1) / kCtaRows;
  const int tiles2 = (d.H + kCtaRows - 1) / kCtaRows;
  const long tch = (Tm + kTokChunk - 1) / kTokChunk;
  const long chunks_routed = std::min<long>(d.E, TK) + TK / kTokChunk + 1;
  c->s.max_items1 = (int)(tiles1 * chunks_routed + (d.Is ? ((2 * d.Is + kCtaRows - 1) / kCtaRows) * tch : 0));
  const int nsplit = shared_down_splits(d.I, d.Is);
  const int dsplit = routed_down_splits(1, d.I);  // the most K parts of a routed down item
  c->s.max_items2 = (int)(tiles2 * chunks_routed * dsplit + (d.Is ? tiles2 * tch * nsplit : 0));
  // routed down partial sums: one part of T*K rows for prefill-sized batches, dsplit parts
  // for decode-sized ones
  const long o_rows = std::max<long>(TK, (long)dsplit * std::min<long>(Tm, kPrefillMinT - 1) * d.K);
  auto salloc = [&](void **p, size_t n) -> bool {
    n = std::max<size_t>(n, 16);
    if (cudaMalloc(p, n) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    c->scratch_allocs.push_back(*p);
    c->scratch_bytes += (int64_t)n;
    return true;
  };
  bool ok = salloc((void **)&c->s.logits, sizeof(float) * Tm * d.E) &&
            salloc((void **)&c->s.ids, sizeof(int) * TK) && salloc((void **)&c->s.w, sizeof(float) * TK) &&
            salloc((void **)&c->s.ranks, sizeof(int) * 4 * kRankStride) &&
            salloc((void **)&c->s.offsets, sizeof(int) * (d.E + 1)) &&
            salloc((void **)&c->s.slot_tok, sizeof(int) * TK) &&
            salloc((void **)&c->s.pair_slot, sizeof(int) * TK) &&
            salloc((void **)&c->s.slot_w, sizeof(float) * TK) &&
            salloc((void **)&c->s.items1, sizeof(WorkItem) * c->s.max_items1) &&
            salloc((void **)&c->s.items2, sizeof(WorkItem) * c->s.max_items2) &&
            salloc((void **)&c->s.n_items, sizeof(int) * 2) && salloc((void **)&c->s.ticket, sizeof(unsigned) * (1 + (Tm + 7) / 8)) &&
            salloc((void **)&c->s.h_routed, sizeof(uint16_t) * TK * d.I) &&
            salloc((void **)&c->s.h_shared, sizeof(uint16_t) * Tm * std::max(d.Is, 1)) &&
            salloc((void **)&c->s.o_routed, sizeof(float) * o_rows * d.H) &&
            salloc((void **)&c->s.o_shared, sizeof(float) * nsplit * Tm * d.H) &&
            salloc((void **)&c->s.inv_rms, sizeof(float) * Tm) && salloc((void **)&c->s.sgate, sizeof(float) * Tm) &&
            salloc((void **)&c->s.xnorm, sizeof(float) * Tm) &&
            salloc((void **)&c->s.stat_phi, sizeof(double) * 4 * d.L * d.E) &&
            salloc((void **)&c->s.xh, sizeof(uint16_t) * Tm * d.H) &&
            salloc((void **)&c->s.err, sizeof(int)) && salloc((void **)&c->s.work, sizeof(int) * 2) &&
            salloc((void **)&c->s.ready, sizeof(int) * 2 * d.L) &&
            salloc((void **)&c->s.stat_count, sizeof(double) * d.L * d.E) &&
            salloc((void **)&c->s.stat_wsum, sizeof(double) * d.L * d.E) &&
            salloc(&c->xdev, sizeof(uint16_t) * Tm * d.H);
  if (ok) ok = salloc((void **)&c->s.xs, sizeof(uint16_t) * TK * d.H);
  if (!ok) {
    fail(nullptr, PW_ERR_OOM, "scratch allocation failed (max_tokens=%d)", d.max_tokens);
    return bail(PW_ERR_OOM);
  }
  {
    bool enc = true;
    for (int k = 0; k < 2; ++k) {
      ActMaps &m = k ? c->bmaps.rows128 : c->bmaps.rows16;
      const unsigned br = k ? 128u : 16u;
      enc = enc && encode_act_map(&m.xs, c->s.xs, TK, d.H, br) && encode_act_map(&m.xh, c->s.xh, Tm, d.H, br) &&
            encode_act_map(&m.h_routed, c->s.h_routed, TK, d.I, br) &&
            (d.Is == 0 || encode_act_map(&m.h_shared, c->s.h_shared, Tm, d.Is, br));
    }
    enc = enc && encode_act_map(&c->bmaps.gemv.xs, c->s.xs, TK, d.H, 8u, 128u) &&
          encode_act_map(&c->bmaps.gemv.h_routed, c->s.h_routed, TK, d.I, 8u, 128u);
    if (!enc) {
      fail(nullptr, PW_ERR_CUDA, "tensor map encoding failed");
      return bail(PW_ERR_CUDA);
    }
    c->has_bmaps = true;
  }
  cudaMemset(c->s.ticket, 0, sizeof(unsigned) * (1 + (Tm + 7) / 8));
  cudaMemset(c->s.err, 0, sizeof(int));
  cudaMemset(c->s.work, 0, sizeof(int) * 2);
  cudaMemset(c->s.ready, 0, sizeof(int) * 2 * d.L);
  cudaMemset(c->s.stat_count, 0, sizeof(double) * d.L * d.E);
  cudaMemset(c->s.stat_wsum, 0, sizeof(double) * d.L * d.E);
  cudaMemset(c->s.stat_phi, 0, sizeof(double) * 4 * d.L * d.E);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    fail(nullptr, PW_ERR_CUDA, "context initialisation failed");
    return bail(PW_ERR_CUDA);
  }
  *out = c;
  return PW_OK;
}

void pw_destroy(pw_ctx *c) {
  if (!c) return;
  cudaSetDevice(c->d.device);
  cudaDeviceSynchronize();
  drop_graphs(c);
  for (auto &b : c->blocks)
    if (b.ev) cudaEventDestroy(b.ev);
  for (auto &l : c->layers) {
    cudaFree(const_cast<float *>(l.Wr));
    cudaFree(const_cast<float *>(l.bias));
    cudaFree(const_cast<uint16_t *>(l.wgu));
    cudaFree(const_cast<uint16_t *>(l.wd));
    cudaFree(const_cast<float *>(l.wsg));
  }
  for (void *p : c->scratch_allocs) cudaFree(p);
  if (c->stage) cudaFree(c->stage);
  if (c->table) cudaFree(c->table);
  if (c->poison) cudaFree(c->poison);
  c->dpool.destroy();
  c->hpool.destroy();
  for (cudaEvent_t e : c->prof_ev) cudaEventDestroy(e);
  if (c->own_compute) cudaStreamDestroy(c->own_compute);
  if (c->io) cudaStreamDestroy(c->io);
  cudaGetLastError();
  delete c;
}

pw_status pw_set_stream(pw_ctx *c, pw_stream stream) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (st != c->compute) {
    // commits already enqueued on the old stream must land before the new one runs
    CU(c, cudaStreamSynchronize(c->compute));
    c->compute = st;
  }
  return PW_OK;
}

pw_status pw_get_stream(pw_ctx *c, pw_stream *stream) {
  if (!c || !stream) return fail(c, PW_ERR_INVALID, "null argument");
  *stream = reinterpret_cast<pw_stream>(c->compute);
  return PW_OK;
}

// ================================================================== weights
pw_status pw_pack(pw_ctx *c, int layer, int expert, int u, const uint8_t *idx, const uint16_t *lut,
                  int q_init) {
  if (!c || !idx || !lut) return fail(c, PW_ERR_INVALID, "null argument");
  if (layer < 0 || layer >= c->d.L || expert < 0 || expert >= c->d.E || (u != 0 && u != 1))
    return fail(c, PW_ERR_INVALID, "block (%d,%d,%d) out of range", layer, expert, u);
  if (!supported(c, q_init)) return fail(c, PW_ERR_INVALID, "q_init=%d is not a supported bitwidth", q_init);
  if (pw_status st = check_sticky(c)) return st;
  cudaSetDevice(c->d.device);
  const int id = (layer * c->d.E + expert) * 2 + u;
  HostBlock &b = c->blocks[id];
  if (pw_status st = observe(c, id)) return st;
  if (b.pend.kind) return fail(c, PW_ERR_BUSY, "block %d has a transfer in flight", id);
  CU(c, cudaStreamSynchronize(c->io));
  CU(c, cudaStreamSynchronize(c->compute));
  const bool on_dev = is_device_ptr(idx);
  if (on_dev != is_device_ptr(lut)) return fail(c, PW_ERR_INVALID, "idx and lut must both be host or both be device memory");

  // release the previous pages of this block
  if (b.packed) {
    for (int p = 0; p < kMaxPlanes; ++p) {
      c->dpool.release(b.dplane[p], b.plane_bytes);
      c->hpool.release(b.hplane[p], b.plane_bytes);
      b.dplane[p] = b.hplane[p] = nullptr;
    }
    for (int bb = 1; bb <= 8; ++bb) {
      c->dpool.release(b.dlut[bb], b.lut_bytes[bb]);
      c->hpool.release(b.hlut[bb], b.lut_bytes[bb]);
      b.dlut[bb] = b.hlut[bb] = nullptr;
    }
    c->packed_count[layer]--;
    b.packed = false;
  }
  // the caller's LUTs: [N][2^b] fp16 per supported b, concatenated
  size_t lut_total = 0;
  for (int i = 0; i < c->n_bits; ++i) lut_total += (size_t)b.N * (1u << c->bits[i]) * 2;
  const size_t idx_bytes = (size_t)b.N * b.K;
  const size_t idx_al = (idx_bytes + 255) & ~size_t(255);
  const size_t lut_al = (lut_total + 255) & ~size_t(255);
  const int bmax = c->d.bmax;
  const size_t planes_tmp = (size_t)bmax * b.plane_bytes;
  const size_t max_lut = b.lut_bytes[8];
  if (pw_status st = ensure_stage(c, idx_al + lut_al + planes_tmp + max_lut + 256)) return st;
  char *stg = static_cast<char *>(c->stage);
  uint8_t *d_idx = reinterpret_cast<uint8_t *>(stg);
  uint16_t *d_lut = reinterpret_cast<uint16_t *>(stg + idx_al);
  char *d_planes_tmp = stg + idx_al + lut_al;
  uint16_t *d_lut_tmp = reinterpret_cast<uint16_t *>(d_planes_tmp + planes_tmp);
  CU(c, cudaMemcpyAsync(d_idx, idx, idx_bytes, cudaMemcpyDefault, c->compute));
  CU(c, cudaMemcpyAsync(d_lut, lut, lut_total, cudaMemcpyDefault, c->compute));

  // allocate the resident pages, stage the rest for the host
  uint32_t *outp[kMaxPlanes];
  for (int p = 0; p < bmax; ++p) {
    if (p < q_init) {
      b.dplane[p] = dev_alloc_page(c, b.plane_bytes);
      if (!b.dplane[p]) return fail(c, PW_ERR_OOM, "device pool exhausted packing block %d", id);
      outp[p] = static_cast<uint32_t *>(b.dplane[p]);
    } else {
      outp[p] = reinterpret_cast<uint32_t *>(d_planes_tmp + (size_t)p * b.plane_bytes);
    }
  }
  uint32_t **d_outp = reinterpret_cast<uint32_t **>(d_lut_tmp + max_lut / 2);
  // the pointer array lives in the staging tail
  CU(c, cudaMemcpyAsync(d_outp, outp, sizeof(outp), cudaMemcpyHostToDevice, c->compute));
  CU(c, cudaStreamSynchronize(c->compute));
  if (int e = launch_pack(d_idx, b.N, b.K, b.KC, u, c->d.I, bmax, d_outp, c->compute))
    return fail(c, PW_ERR_CUDA, "pack kernel: %s", cudaGetErrorString((cudaError_t)e));
  for (int p = q_init; p < bmax; ++p) {
    b.hplane[p] = c->hpool.alloc(b.plane_bytes);
    if (!b.hplane[p]) return fail(c, PW_ERR_OOM, "pinned host pool exhausted packing block %d", id);
    CU(c, cudaMemcpyAsync(b.hplane[p], outp[p], b.plane_bytes, cudaMemcpyDeviceToHost, c->compute));
    CU(c, cudaStreamSynchronize(c->compute));
  }
  size_t off = 0;
  for (int i = 0; i < c->n_bits; ++i) {
    const int bb = c->bits[i];
    const uint16_t *src = d_lut + off / 2;
    off += (size_t)b.N * (1u << bb) * 2;
    if (bb <= q_init) {
      b.dlut[bb] = dev_alloc_page(c, b.lut_bytes[bb]);
      if (!b.dlut[bb]) return fail(c, PW_ERR_OOM, "device pool exhausted packing block %d", id);
      if (int e = launch_lut_permute(src, b.N, 1 << bb, u, c->d.I, static_cast<uint16_t *>(b.dlut[bb]), c->compute))
        return fail(c, PW_ERR_CUDA, "lut kernel: %s", cudaGetErrorString((cudaError_t)e));
    } else {
      if (int e = launch_lut_permute(src, b.N, 1 << bb, u, c->d.I, d_lut_tmp, c->compute))
        return fail(c, PW_ERR_CUDA, "lut kernel: %s", cudaGetErrorString((cudaError_t)e));
      b.hlut[bb] = c->hpool.alloc(b.lut_bytes[bb]);
      if (!b.hlut[bb]) return fail(c, PW_ERR_OOM, "pinned host pool exhausted packing block %d", id);
      CU(c, cudaMemcpyAsync(b.hlut[bb], d_lut_tmp, b.lut_bytes[bb], cudaMemcpyDeviceToHost, c->compute));
      CU(c, cudaStreamSynchronize(c->compute));
    }
  }
  for (int p = 0; p < kMaxPlanes; ++p) b.state[p] = (p < q_init) ? PW_PAGE_GPU : PW_PAGE_CPU;
  b.q = b.d = b.q_init = q_init;
  b.pend = Pending{};
  b.packed = true;
  c->packed_count[layer]++;
  if (int e = launch_commit(c->table, id, dev_entry(c, b, q_init), c->compute))
    return fail(c, PW_ERR_CUDA, "commit kernel: %s", cudaGetErrorString((cudaError_t)e));
  CU(c, cudaStreamSynchronize(c->compute));
  return PW_OK;
}

pw_status pw_set_router(pw_ctx *c, int layer, const float *Wr, const float *bias) {
  if (!c || !Wr) return fail(c, PW_ERR_INVALID, "null argument");
  if (layer < 0 || layer >= c->d.L) return fail(c, PW_ERR_INVALID, "layer out of range");
  cudaSetDevice(c->d.device);
  LayerDev &l = c->layers[layer];
  const size_t n = sizeof(float) * c->d.E * c->d.H;
  CU(c, cudaStreamSynchronize(c->compute));
  if (!l.Wr) CU(c, cudaMalloc((void **)&l.Wr, n));
  CU(c, cudaMemcpy(const_cast<float *>(l.Wr), Wr, n, cudaMemcpyDefault));
  if (bias) {
    if (!l.bias) CU(c, cudaMalloc((void **)&l.bias, sizeof(float) * c->d.E));
    CU(c, cudaMemcpy(const_cast<float *>(l.bias), bias, sizeof(float) * c->d.E, cudaMemcpyDefault));
  } else if (l.bias) {
    cudaFree(const_cast<float *>(l.bias));
    l.bias = nullptr;
    drop_graphs(c);
  }
  c->router_set[layer] = 1;
  return PW_OK;
}

pw_status pw_set_shared(pw_ctx *c, int layer, const uint16_t *wgu, const uint16_t *wd) {
  if (!c || !wgu || !wd) return fail(c, PW_ERR_INVALID, "null argument");
  if (layer < 0 || layer >= c->d.L) return fail(c, PW_ERR_INVALID, "layer out of range");
  if (c->d.Is == 0) return fail(c, PW_ERR_INVALID, "this context has no shared expert (Is = 0)");
  cudaSetDevice(c->d.device);
  LayerDev &l = c->layers[layer];
  const int H = c->d.H, Is = c->d.Is;
  const size_t ngu = sizeof(uint16_t) * 2 * (size_t)Is * H, nd = sizeof(uint16_t) * (size_t)H * Is;
  // device copies: rows and columns padded to multiples of 128 (operand tiles), zero-filled
  auto pad128 = [](size_t n) { return (n + 127) / 128 * 128; };
  const size_t dgu = sizeof(uint16_t) * pad128(2 * (size_t)Is) * pad128(H);
  const size_t dd = sizeof(uint16_t) * pad128(H) * pad128(Is);
  CU(c, cudaStreamSynchronize(c->compute));
  if (!l.wgu) CU(c, cudaMalloc((void **)&l.wgu, dgu));
  if (!l.wd) CU(c, cudaMalloc((void **)&l.wd, dd));
  CU(c, cudaMemsetAsync(const_cast<uint16_t *>(l.wgu), 0, dgu, c->compute));
  CU(c, cudaMemsetAsync(const_cast<uint16_t *>(l.wd), 0, dd, c->compute));
  if (pw_status st = ensure_stage(c, std::max(ngu, nd) + 256)) return st;
  int *d_bad = reinterpret_cast<int *>(static_cast<char *>(c->stage) + std::max(ngu, nd));
  CU(c, cudaMemsetAsync(d_bad, 0, sizeof(int), c->compute));
  CU(c, cudaMemcpyAsync(c->stage, wgu, ngu, cudaMemcpyDefault, c->compute));
  if (int e = launch_frag16(static_cast<uint16_t *>(c->stage), 2 * Is, H, 0, Is, const_cast<uint16_t *>(l.wgu), d_bad, c->compute))
    return fail(c, PW_ERR_CUDA, "frag16 kernel: %s", cudaGetErrorString((cudaError_t)e));
  CU(c, cudaMemcpyAsync(c->stage, wd, nd, cudaMemcpyDefault, c->compute));
  if (int e = launch_frag16(static_cast<uint16_t *>(c->stage), H, Is, 1, Is, const_cast<uint16_t *>(l.wd), d_bad, c->compute))
    return fail(c, PW_ERR_CUDA, "frag16 kernel: %s", cudaGetErrorString((cudaError_t)e));
  int bad = 0;
  CU(c, cudaMemcpyAsync(&bad, d_bad, sizeof(int), cudaMemcpyDeviceToHost, c->compute));
  CU(c, cudaStreamSynchronize(c->compute));
  if (bad) return fail(c, PW_ERR_INVALID, "%d shared-expert weights exceed the fp16 range (|w| > 65504)", bad);
  c->shared_set[layer] = 1;
  return PW_OK;
}

pw_status pw_set_shared_gate(pw_ctx *c, int layer, const float *wsg) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (layer < 0 || layer >= c->d.L) return fail(c, PW_ERR_INVALID, "layer out of range");
  if (c->d.Is == 0) return fail(c, PW_ERR_INVALID, "this context has no shared expert (Is = 0)");
  cudaSetDevice(c->d.device);
  LayerDev &l = c->layers[layer];
  CU(c, cudaStreamSynchronize(c->compute));  // no launch in flight reads the old gate
  if (!wsg) {
    cudaFree(const_cast<float *>(l.wsg));
    l.wsg = nullptr;
    drop_graphs(c);  // captured launches hold the old layer description
    return PW_OK;
  }
  if (!l.wsg) {
    CU(c, cudaMalloc((void **)&l.wsg, sizeof(float) * c->d.H));
    drop_graphs(c);
  }
  CU(c, cudaMemcpyAsync(const_cast<float *>(l.wsg), wsg, sizeof(float) * c->d.H, cudaMemcpyDefault, c->compute));
  CU(c, cudaStreamSynchronize(c->compute));
  return PW_OK;
}

// ================================================================== forward
static pw_status forward_args(pw_ctx *c, int layer, const void *x, int T, void *y, int32_t *ids, float *w,
                              int flags, FwdArgs *a) {
  if (layer < 0 || layer >= c->d.L) return fail(c, PW_ERR_INVALID, "layer out of range");
  if (T < 1 || T > c->d.max_tokens) return fail(c, PW_ERR_INVALID, "T=%d outside 1..max_tokens=%d", T, c->d.max_tokens);
  if (!x || !y) return fail(c, PW_ERR_INVALID, "null x or y");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15)
    return fail(c, PW_ERR_INVALID, "x and y must be 16-byte aligned");
  if (!c->router_set[layer]) return fail(c, PW_ERR_STATE, "router of layer %d not set", layer);
  if (c->d.Is && !c->shared_set[layer]) return fail(c, PW_ERR_STATE, "shared expert of layer %d not set", layer);
  if (c->packed_count[layer] != 2 * c->d.E) return fail(c, PW_ERR_STATE, "layer %d has unpacked blocks", layer);
  *a = FwdArgs{};
  a->layer = layer;
  a->stat_layer = layer;
  a->T = T;
  a->E = c->d.E;
  a->H = c->d.H;
  a->I = c->d.I;
  a->K = c->d.K;
  a->Is = c->d.Is;
  a->renorm = c->d.renorm;
  a->flags = flags;
  a->table = c->table;
  a->lay = c->layers[layer];
  a->s = c->s;
  a->x = static_cast<const uint16_t *>(x);
  a->y = static_cast<uint16_t *>(y);
  a->ids_out = ids;
  a->w_out = w;
  a->sm_count = c->sm_count;
  a->gemv_max = c->gemv_max;
  a->wait_cycles = c->wait_cycles;
  a->withhold = c->fault_withhold;
  c->fault_withhold = 0;  // one launch
  a->bmaps = c->has_bmaps ? &c->bmaps : nullptr;
  return PW_OK;
}

pw_status pw_moe_forward(pw_ctx *c, int layer, const void *x, int T, void *y, int32_t *ids, float *w, int flags,
                         pw_stream stream) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (pw_status st = check_sticky(c)) return st;
  FwdArgs a;
  if (pw_status st = forward_args(c, layer, x, T, y, ids, w, flags, &a)) return st;
  if (int e = launch_forward(a, stream, c->profiling ? reinterpret_cast<void *const *>(&c->prof_ev[(size_t)layer * 5]) : nullptr)) {
    c->sticky = 1;
    return fail(c, PW_ERR_CUDA, "forward launch failed: %s", cudaGetErrorString((cudaError_t)e));
  }
  return PW_OK;
}

static pw_status stack_launch(pw_ctx *c, void *x, int T, cudaStream_t st) {
  for (int l = 0; l < c->d.L; ++l) {
    FwdArgs a;
    if (pw_status s = forward_args(c, l, x, T, x, nullptr, nullptr, PW_ACCUMULATE | PW_PRENORM, &a)) return s;
    if (int e = launch_forward(a, st, c->profiling ? reinterpret_cast<void *const *>(&c->prof_ev[(size_t)l * 5]) : nullptr))
      return fail(c, PW_ERR_CUDA, "forward launch failed: %s", cudaGetErrorString((cudaError_t)e));
  }
  return PW_OK;
}

pw_status pw_stack_forward(pw_ctx *c, void *x, int T, pw_stream stream) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (pw_status st = check_sticky(c)) return st;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!st) return stack_launch(c, x, T, st);  // the legacy stream cannot be captured
  for (auto &g : c->graphs)
    if (g.x == x && g.T == T && g.stream == st && g.profiling == c->profiling) {
      CU(c, cudaGraphLaunch(g.exec, st));
      return PW_OK;
    }
  // validate everything before capturing
  for (int l = 0; l < c->d.L; ++l) {
    FwdArgs a;
    if (pw_status s = forward_args(c, l, x, T, x, nullptr, nullptr, PW_ACCUMULATE | PW_PRENORM, &a)) return s;
  }
  CU(c, cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
  pw_status s = stack_launch(c, x, T, st);
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamEndCapture(st, &graph);
  if (s != PW_OK) {
    if (graph) cudaGraphDestroy(graph);
    return s;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(c, PW_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
  }
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(c, PW_ERR_CUDA, "graph instantiation failed: %s", cudaGetErrorString(e));
  }
  c->graphs.push_back(GraphEntry{x, T, c->profiling, st, exec});
  CU(c, cudaGraphLaunch(exec, st));
  return PW_OK;
}

pw_status pw_stack_forward_host(pw_ctx *c, const void *x_host, int T, void *y_host) {
  if (!c || !x_host || !y_host) return fail(c, PW_ERR_INVALID, "null argument");
  if (T < 1 || T > c->d.max_tokens) return fail(c, PW_ERR_INVALID, "T out of range");
  const size_t n = sizeof(uint16_t) * (size_t)T * c->d.H;
  CU(c, cudaMemcpyAsync(c->xdev, x_host, n, cudaMemcpyHostToDevice, c->compute));
  if (pw_status st = pw_stack_forward(c, c->xdev, T, c->compute)) return st;
  CU(c, cudaMemcpyAsync(y_host, c->xdev, n, cudaMemcpyDeviceToHost, c->compute));
  CU(c, cudaStreamSynchronize(c->compute));
  return check_sticky(c);
}

pw_status pw_routing_stats(pw_ctx *c, int layer, double *count, double *weight_sum, int reset) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (layer < 0 || layer >= c->d.L) return fail(c, PW_ERR_INVALID, "layer out of range");
  CU(c, cudaStreamSynchronize(c->compute));
  const size_t off = (size_t)layer * c->d.E;
  if (count) CU(c, cudaMemcpy(count, c->s.stat_count + off, sizeof(double) * c->d.E, cudaMemcpyDeviceToHost));
  if (weight_sum) CU(c, cudaMemcpy(weight_sum, c->s.stat_wsum + off, sizeof(double) * c->d.E, cudaMemcpyDeviceToHost));
  if (reset) {
    CU(c, cudaMemset(c->s.stat_count + off, 0, sizeof(double) * c->d.E));
    CU(c, cudaMemset(c->s.stat_wsum + off, 0, sizeof(double) * c->d.E));
  }
  return check_sticky(c);
}

// Eq. 5 features of `layer`'s experts from the device sums: phi[e] = (sum r n / sum r,
// sqrt(sum r n^2 / sum r), max n), zeros where no token was routed.
static pw_status read_features(pw_ctx *c, int layer, double *phi, int reset) {
  const int E = c->d.E;
  std::vector<double> raw((size_t)4 * E);
  const size_t off = (size_t)layer * E * 4;
  CU(c, cudaMemcpy(raw.data(), c->s.stat_phi + off, sizeof(double) * 4 * E, cudaMemcpyDeviceToHost));
  for (int e = 0; e < E; ++e) {
    const double *r = &raw[(size_t)e * 4];
    double *o = phi + (size_t)e * 3;
    if (r[0] > 0) {
      o[0] = r[1] / r[0];
      o[1] = std::sqrt(r[2] / r[0]);
      o[2] = r[3];
    } else {
      o[0] = o[1] = o[2] = 0.0;
    }
  }
  if (reset) CU(c, cudaMemset(c->s.stat_phi + off, 0, sizeof(double) * 4 * E));
  return PW_OK;
}

pw_status pw_routing_features(pw_ctx *c, int layer, double *phi, int reset) {
  if (!c || !phi) return fail(c, PW_ERR_INVALID, "null argument");
  if (layer < 0 || layer >= c->d.L) return fail(c, PW_ERR_INVALID, "layer out of range");
  CU(c, cudaStreamSynchronize(c->compute));
  if (pw_status st = read_features(c, layer, phi, reset)) return st;
  return check_sticky(c);
}

// ================================================================== page table
pw_status pw_set_bits(pw_ctx *c, int block, int q) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (block < 0 || block >= (int)c->blocks.size()) return fail(c, PW_ERR_INVALID, "block out of range");
  if (pw_status st = observe(c, block)) return st;
  HostBlock &b = c->blocks[block];
  if (!b.packed) return fail(c, PW_ERR_STATE, "block %d is not packed", block);
  if (!supported(c, q)) return fail(c, PW_ERR_INVALID, "bitwidth %d not supported", q);
  if (b.pend.kind) return fail(c, PW_ERR_BUSY, "block %d has a transfer in flight", block);
  for (int p = 0; p < q; ++p)
    if (b.state[p] != PW_PAGE_GPU) return fail(c, PW_ERR_STATE, "page %d of block %d is not GPU-resident", p, block);
  if (int e = launch_commit(c->table, block, dev_entry(c, b, q), c->compute))
    return fail(c, PW_ERR_CUDA, "commit kernel: %s", cudaGetErrorString((cudaError_t)e));
  b.q = b.d = q;
  return PW_OK;
}

static bool copy_fault(pw_ctx *c) { return c->fault_copy > 0 && --c->fault_copy == 0; }

pw_status pw_offload(pw_ctx *c, int block, int q_new) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (block < 0 || block >= (int)c->blocks.size()) return fail(c, PW_ERR_INVALID, "block out of range");
  if (pw_status st = observe(c, block)) return st;
  if (pw_status st = check_sticky(c)) return st;
  HostBlock &b = c->blocks[block];
  if (!b.packed) return fail(c, PW_ERR_STATE, "block %d is not packed", block);
  if (b.pend.kind) return fail(c, PW_ERR_BUSY, "block %d has a transfer in flight", block);
  if (!supported(c, q_new) || q_new >= b.q)
    return fail(c, PW_ERR_STATE, "offload of block %d needs a supported bitwidth below q=%d (got %d)", block, b.q, q_new);
  for (int p = q_new; p < b.q; ++p)
    if (b.state[p] != PW_PAGE_GPU) return fail(c, PW_ERR_STATE, "page %d of block %d is not GPU-resident", p, block);
  // host slots first, so that a pinned-memory shortage changes nothing
  for (int p = q_new; p < b.q; ++p)
    if (!b.hplane[p] && !(b.hplane[p] = c->hpool.alloc(b.plane_bytes)))
      return fail(c, PW_ERR_OOM, "pinned host pool exhausted");
  for (int i = 0; i < c->n_bits; ++i) {
    const int bb = c->bits[i];
    if (bb > q_new && bb <= b.q && !b.hlut[bb] && !(b.hlut[bb] = c->hpool.alloc(b.lut_bytes[bb])))
      return fail(c, PW_ERR_OOM, "pinned host pool exhausted");
  }
  const int q_old = b.q;
  // 1. lower the committed bitwidth on the compute stream
  if (int e = launch_commit(c->table, block, dev_entry(c, b, q_new), c->compute))
    return fail(c, PW_ERR_CUDA, "commit kernel: %s", cudaGetErrorString((cudaError_t)e));
  b.q = b.d = q_new;
  // 2. move the pages once the compute stream has passed the lowering
  CU(c, cudaEventRecord(b.ev, c->compute));
  CU(c, cudaStreamWaitEvent(c->io, b.ev, 0));
  bool failed = false;
  for (int p = q_new; p < q_old; ++p) {
    if (copy_fault(c)) {
      failed = true;
      continue;
    }
    CU(c, cudaMemcpyAsync(b.hplane[p], b.dplane[p], b.plane_bytes, cudaMemcpyDeviceToHost, c->io));
  }
  for (int i = 0; i < c->n_bits; ++i) {
    const int bb = c->bits[i];
    if (bb > q_new && bb <= q_old) {
      if (copy_fault(c)) {
        failed = true;
        continue;
      }
      CU(c, cudaMemcpyAsync(b.hlut[bb], b.dlut[bb], b.lut_bytes[bb], cudaMemcpyDeviceToHost, c->io));
    }
  }
  CU(c, cudaEventRecord(b.ev, c->io));
  for (int p = q_new; p < q_old; ++p) b.state[p] = PW_PAGE_TO_CPU;
  b.pend = Pending{1, q_old, q_new, failed};
  return PW_OK;
}

pw_status pw_reload(pw_ctx *c, int block, int q_new) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (block < 0 || block >= (int)c->blocks.size()) return fail(c, PW_ERR_INVALID, "block out of range");
  if (pw_status st = observe(c, block)) return st;
  if (pw_status st = check_sticky(c)) return st;
  HostBlock &b = c->blocks[block];
  if (!b.packed) return fail(c, PW_ERR_STATE, "block %d is not packed", block);
  if (b.pend.kind) return fail(c, PW_ERR_BUSY, "block %d has a transfer in flight", block);
  if (!supported(c, q_new) || q_new <= b.q)
    return fail(c, PW_ERR_STATE, "reload of block %d needs a supported bitwidth above q=%d (got %d)", block, b.q, q_new);
  for (int p = b.q; p < q_new; ++p)
    if (b.state[p] != PW_PAGE_CPU && b.state[p] != PW_PAGE_GPU)
      return fail(c, PW_ERR_STATE, "page %d of block %d is in transfer", p, block);
  // allocate every device page first; on failure give them back and change nothing
  std::vector<std::pair<void **, size_t>> got;
  auto undo = [&]() {
    for (auto &g : got) {
      c->dpool.release(*g.first, g.second);
      *g.first = nullptr;
    }
  };
  for (int p = b.q; p < q_new; ++p) {
    if (b.state[p] == PW_PAGE_CPU) {
      b.dplane[p] = dev_alloc_page(c, b.plane_bytes);
      if (!b.dplane[p]) {
        undo();
        return fail(c, PW_ERR_OOM, "device pool exhausted reloading block %d", block);
      }
      got.push_back({&b.dplane[p], b.plane_bytes});
    }
  }
  unsigned new_luts = 0;
  for (int i = 0; i < c->n_bits; ++i) {
    const int bb = c->bits[i];
    if (bb > b.q && bb <= q_new && !b.dlut[bb]) {
      b.dlut[bb] = dev_alloc_page(c, b.lut_bytes[bb]);
      if (!b.dlut[bb]) {
        undo();
        return fail(c, PW_ERR_OOM, "device pool exhausted reloading block %d", block);
      }
      got.push_back({&b.dlut[bb], b.lut_bytes[bb]});
      new_luts |= 1u << bb;
    }
  }
  bool failed = false;
  for (int p = b.q; p < q_new; ++p) {
    if (b.state[p] != PW_PAGE_CPU) continue;
    if (copy_fault(c)) {
      failed = true;
    } else {
      CU(c, cudaMemcpyAsync(b.dplane[p], b.hplane[p], b.plane_bytes, cudaMemcpyHostToDevice, c->io));
    }
    b.state[p] = PW_PAGE_TO_GPU;
  }
  for (int bb = 1; bb <= 8; ++bb) {
    if (!((new_luts >> bb) & 1u)) continue;
    if (copy_fault(c)) {
      failed = true;
      continue;
    }
    CU(c, cudaMemcpyAsync(b.dlut[bb], b.hlut[bb], b.lut_bytes[bb], cudaMemcpyHostToDevice, c->io));
  }
  CU(c, cudaEventRecord(b.ev, c->io));
  b.pend = Pending{2, b.q, q_new, failed, new_luts};
  b.d = q_new;
  return PW_OK;
}

// Host-side observation of a block's transfer (never blocks).  A landed offload retires
// its device pages; a landed reload makes its pages GPU-resident but leaves q alone (the
// raise is pw_commit's).  A failed transfer is rolled back and remembered in io_error.
}  // extern "C"

namespace {
pw_status observe(pw_ctx *c, int id) {
  HostBlock &b = c->blocks[id];
  if (!b.pend.kind || b.landed || c->hold) return PW_OK;
  cudaError_t e = cudaEventQuery(b.ev);
  if (e == cudaErrorNotReady) return PW_OK;
  if (e != cudaSuccess) {
    c->sticky = 1;
    return fail(c, PW_ERR_CUDA, "page copy of block %d failed: %s", id, cudaGetErrorString(e));
  }
  const Pending pd = b.pend;
  if (pd.kind == 1) {  // offload landed
    b.pend = Pending{};
    if (pd.failed) {
      for (int p = pd.to; p < pd.from; ++p) b.state[p] = PW_PAGE_GPU;  // pages stay; q stays lowered
      b.io_error = 1;
      return PW_OK;
    }
    for (int p = pd.to; p < pd.from; ++p) {
      if (c->d.flags & PW_FLAG_POISON) cudaMemsetAsync(b.dplane[p], 0xFF, b.plane_bytes, c->io);
      c->dpool.release(b.dplane[p], b.plane_bytes);
      b.dplane[p] = nullptr;
      b.state[p] = PW_PAGE_CPU;
    }
    for (int i = 0; i < c->n_bits; ++i) {
      const int bb = c->bits[i];
      if (bb > pd.to && bb <= pd.from && b.dlut[bb]) {
        if (c->d.flags & PW_FLAG_POISON) cudaMemsetAsync(b.dlut[bb], 0xFF, b.lut_bytes[bb], c->io);
        c->dpool.release(b.dlut[bb], b.lut_bytes[bb]);
        b.dlut[bb] = nullptr;
      }
    }
    return PW_OK;
  }
  // reload landed
  if (pd.failed) {
    b.pend = Pending{};
    for (int p = pd.from; p < pd.to; ++p) {
      if (b.state[p] == PW_PAGE_TO_GPU) {
        c->dpool.release(b.dplane[p], b.plane_bytes);
        b.dplane[p] = nullptr;
        b.state[p] = PW_PAGE_CPU;
      }
    }
    for (int bb = 1; bb <= 8; ++bb) {
      if ((pd.new_luts >> bb) & 1u) {
        c->dpool.release(b.dlut[bb], b.lut_bytes[bb]);
        b.dlut[bb] = nullptr;
      }
    }
    b.d = b.q;
    b.io_error = 2;
    return PW_OK;
  }
  for (int p = pd.from; p < pd.to; ++p) b.state[p] = PW_PAGE_GPU;
  b.landed = true;
  return PW_OK;
}
}  // namespace

extern "C" {

pw_status pw_commit(pw_ctx *c, int *n_applied) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (n_applied) *n_applied = 0;
  if (pw_status st = check_sticky(c)) return st;
  int applied = 0;
  pw_status result = PW_OK;
  for (int id = 0; id < (int)c->blocks.size(); ++id) {
    HostBlock &b = c->blocks[id];
    if (pw_status st = observe(c, id)) return st;
    if (b.io_error) {
      result = fail(c, PW_ERR_CUDA, b.io_error == 1 ? "offload copy of block %d failed; pages kept on the GPU"
                                                     : "reload copy of block %d failed; bitwidth not raised", id);
      b.io_error = 0;
      continue;
    }
    if (b.pend.kind == 2 && b.landed) {
      const int to = b.pend.to;
      b.pend = Pending{};
      b.landed = false;
      CU(c, cudaStreamWaitEvent(c->compute, b.ev, 0));
      if (int ee = launch_commit(c->table, id, dev_entry(c, b, to), c->compute))
        return fail(c, PW_ERR_CUDA, "commit kernel: %s", cudaGetErrorString((cudaError_t)ee));
      b.q = to;
      ++applied;
    }
  }
  if (n_applied) *n_applied = applied;
  return result;
}

pw_status pw_sync_io(pw_ctx *c) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  CU(c, cudaStreamSynchronize(c->io));
  return check_sticky(c);
}

pw_status pw_query(pw_ctx *c, int block, pw_block_info *info) {
  if (!c || !info) return fail(c, PW_ERR_INVALID, "null argument");
  if (block < 0 || block >= (int)c->blocks.size()) return fail(c, PW_ERR_INVALID, "block out of range");
  if (pw_status st = observe(c, block)) return st;
  const HostBlock &b = c->blocks[block];
  *info = pw_block_info{};
  info->layer = b.layer;
  info->expert = b.expert;
  info->u = b.u;
  info->N = b.N;
  info->K = b.K;
  info->q = b.packed ? b.q : 0;
  info->d = b.packed ? b.d : 0;
  info->pending_q = b.pend.kind == 2 ? b.pend.to : 0;
  for (int p = 0; p < 8; ++p) info->state[p] = (p < c->d.bmax) ? b.state[p] : PW_PAGE_CPU;
  for (int bb = 0; bb <= 8; ++bb) info->M[bb] = supported(c, bb) ? block_M(c, b, bb) : -1;
  return PW_OK;
}

pw_status pw_memory(pw_ctx *c, pw_mem_info *info) {
  if (!c || !info) return fail(c, PW_ERR_INVALID, "null argument");
  *info = pw_mem_info{};
  for (const auto &b : c->blocks) {
    if (!b.packed) continue;
    info->resident_bytes += block_M(c, b, b.q);
    for (int p = 0; p < kMaxPlanes; ++p)
      if (b.dplane[p]) info->held_bytes += (int64_t)b.plane_bytes;
    for (int bb = 1; bb <= 8; ++bb)
      if (b.dlut[bb]) info->held_bytes += (int64_t)b.lut_bytes[bb];
  }
  info->device_pool_bytes = c->dpool.reserved;
  info->device_pool_free = c->dpool.free_bytes;
  info->pinned_bytes = c->hpool.reserved;
  info->scratch_bytes = c->scratch_bytes;
  return PW_OK;
}

pw_status pw_set_fault(pw_ctx *c, int kind, int n) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (kind == 1)
    c->fault_copy = n;
  else if (kind == 2)
    c->fault_alloc = n;
  else if (kind == 3)
    c->hold = n ? 1 : 0;
  else if (kind == 4)
    c->fault_withhold = n ? 1 : 0;
  else if (kind == 5) {
    if (n < 0) return fail(c, PW_ERR_INVALID, "wait limit must be >= 0 microseconds");
    c->wait_cycles = n ? (long long)n * 2000 : kWaitCyclesDefault;  // about 2 SM cycles per ns
  } else
    return fail(c, PW_ERR_INVALID, "unknown fault kind %d", kind);
  if (kind >= 4) drop_graphs(c);  // captured launches hold the old arguments
  return PW_OK;
}

// ================================================================== inspection
static pw_status readback(pw_ctx *c, int block, int b, uint8_t *idx_out, uint16_t *w_out) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (block < 0 || block >= (int)c->blocks.size()) return fail(c, PW_ERR_INVALID, "block out of range");
  if (pw_status st = observe(c, block)) return st;
  HostBlock &hb = c->blocks[block];
  if (!hb.packed) return fail(c, PW_ERR_STATE, "block %d is not packed", block);
  if (b < 1 || b > c->d.bmax) return fail(c, PW_ERR_INVALID, "bitwidth out of range");
  for (int p = 0; p < b; ++p)
    if (hb.state[p] != PW_PAGE_GPU) return fail(c, PW_ERR_STATE, "page %d is not GPU-resident", p);
  if (w_out && (!supported(c, b) || !hb.dlut[b])) return fail(c, PW_ERR_STATE, "LUT_%d is not GPU-resident", b);
  if (pw_status st = check_sticky(c)) return st;
  const size_t n = (size_t)hb.N * hb.K;
  const size_t out_al = (n * 2 + 255) & ~size_t(255);
  CU(c, cudaStreamSynchronize(c->compute));
  // output area, then a private table row whose bitwidth is b, so that the kernel reads
  // exactly planes 0..b-1 and LUT_b
  if (pw_status st = ensure_stage(c, out_al + sizeof(BlockDev))) return st;
  char *stg = static_cast<char *>(c->stage);
  BlockDev *drow = reinterpret_cast<BlockDev *>(stg + out_al);
  BlockDev v = dev_entry(c, hb, c->d.bmax);
  v.q = b;
  CU(c, cudaMemcpy(drow, &v, sizeof v, cudaMemcpyHostToDevice));
  if (int e = launch_unpack(drow, 0, b, hb.u, c->d.I, hb.N, hb.KC, idx_out ? reinterpret_cast<uint8_t *>(stg) : nullptr,
                            w_out ? reinterpret_cast<uint16_t *>(stg) : nullptr, c->compute))
    return fail(c, PW_ERR_CUDA, "unpack kernel: %s", cudaGetErrorString((cudaError_t)e));
  CU(c, cudaStreamSynchronize(c->compute));
  if (idx_out) CU(c, cudaMemcpy(idx_out, stg, n, cudaMemcpyDeviceToHost));
  if (w_out) CU(c, cudaMemcpy(w_out, stg, n * 2, cudaMemcpyDeviceToHost));
  return check_sticky(c);
}

pw_status pw_unpack_indices(pw_ctx *c, int block, int b, uint8_t *host_out) {
  if (!host_out) return fail(c, PW_ERR_INVALID, "null output");
  return readback(c, block, b, host_out, nullptr);
}

pw_status pw_dequant(pw_ctx *c, int block, int b, uint16_t *host_out) {
  if (!host_out) return fail(c, PW_ERR_INVALID, "null output");
  return readback(c, block, b, nullptr, host_out);
}

// ================================================================== planner on the context
pw_status pw_plan_step(pw_ctx *c, const pw_obs *obs, const pw_offline *off, pw_plan *out) {
  if (!c || !obs || !off || !out) return fail(c, PW_ERR_INVALID, "null argument");
  if (off->n_bits != c->n_bits) return fail(c, PW_ERR_INVALID, "offline table has %d bitwidths, context %d", off->n_bits, c->n_bits);
  std::vector<double> dev_phi;  // obs->phi == NULL: the device's routed-input features (Eq. 5)
  if (!obs->phi && !obs->rho_hat) {
    CU(c, cudaStreamSynchronize(c->compute));
    std::vector<double> lay((size_t)c->d.E * 3);
    dev_phi.resize(c->blocks.size() * 3);
    for (int l = 0; l < c->d.L; ++l) {
      if (pw_status st = read_features(c, l, lay.data(), 0)) return st;
      for (size_t i = 0; i < c->blocks.size(); ++i)
        if (c->blocks[i].layer == l)
          for (int j = 0; j < 3; ++j) dev_phi[i * 3 + j] = lay[(size_t)c->blocks[i].expert * 3 + j];
    }
  }
  const double *obs_phi = obs->phi ? obs->phi : dev_phi.empty() ? nullptr : dev_phi.data();
  const int nb = c->n_bits, L = c->d.L, E = c->d.E;
  // A block whose pages are still in transfer (or whose landed reload awaits pw_commit)
  // cannot take another step yet: the problem holds the idle blocks only.
  std::vector<int> ids;
  for (int i = 0; i < (int)c->blocks.size(); ++i) {
    if (!c->blocks[i].packed) return fail(c, PW_ERR_STATE, "block %d is not packed", i);
    if (pw_status st = observe(c, i)) return st;
    if (!c->blocks[i].pend.kind) ids.push_back(i);
  }
  const int n = (int)ids.size();
  std::vector<int> q(n), q0(n), ut(n), ly(n), ex(n);
  std::vector<double> M((size_t)n * nb), phi((size_t)n * 3), rho(obs->rho_hat ? (size_t)n * (nb - 1) : 0);
  for (int k = 0; k < n; ++k) {
    const HostBlock &b = c->blocks[ids[k]];
    q[k] = b.q;
    q0[k] = b.q_init;
    ut[k] = b.u;
    ly[k] = b.layer;
    ex[k] = b.expert;
    for (int j = 0; j < nb; ++j) M[(size_t)k * nb + j] = (double)block_M(c, b, c->bits[j]);
    if (obs_phi)
      for (int j = 0; j < 3; ++j) phi[(size_t)k * 3 + j] = obs_phi[(size_t)ids[k] * 3 + j];
    if (obs->rho_hat)
      for (int j = 0; j < nb - 1; ++j) rho[(size_t)k * (nb - 1) + j] = obs->rho_hat[(size_t)ids[k] * (nb - 1) + j];
  }
  std::vector<double> mass;
  pw_obs o = *obs;
  o.phi = obs_phi ? phi.data() : nullptr;
  o.rho_hat = obs->rho_hat ? rho.data() : nullptr;
  if (!o.mass) {  // Eq. 1 from the online routing statistics
    CU(c, cudaStreamSynchronize(c->compute));
    mass.resize((size_t)L * E);
    CU(c, cudaMemcpy(mass.data(), c->s.stat_wsum, sizeof(double) * L * E, cudaMemcpyDeviceToHost));
    for (int l = 0; l < L; ++l) {
      double tot = 0.0;
      for (int e = 0; e < E; ++e) tot += mass[(size_t)l * E + e];
      for (int e = 0; e < E; ++e) mass[(size_t)l * E + e] = tot > 0 ? mass[(size_t)l * E + e] / tot : 1.0 / E;
    }
    o.mass = mass.data();
  }
  // the offline sensitivities are per block too: the idle blocks' rows
  if (!off->s) return fail(c, PW_ERR_INVALID, "off->s is required");
  std::vector<double> s_sub((size_t)n * nb);
  for (int k = 0; k < n; ++k)
    for (int j = 0; j < nb; ++j) s_sub[(size_t)k * nb + j] = off->s[(size_t)ids[k] * nb + j];
  pw_offline off_sub = *off;
  off_sub.s = s_sub.data();
  pw_plan_problem prob{n, nb, L, E, c->bits, q.data(), q0.data(), ut.data(), ly.data(), ex.data(), M.data()};
  pw_status st = pw_plan_host(&prob, &o, &off_sub, out);
  if (st != PW_OK) return fail(c, st, "planner rejected its inputs (or the plan did not fit in out->capacity)");
  for (int k = 0; k < out->n; ++k) {
    out->entries[k].block = ids[out->entries[k].block];
    c->blocks[out->entries[k].block].d = out->entries[k].to_bits;
  }
  return PW_OK;
}

// ================================================================== decode kernel choice
pw_status pw_set_gemv_tokens(pw_ctx *c, int max_tokens) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (max_tokens < 0 || max_tokens > kGemvMaxTokens)
    return fail(c, PW_ERR_INVALID, "GEMV token threshold %d outside 0..%d", max_tokens, kGemvMaxTokens);
  if (c->gemv_max != max_tokens) drop_graphs(c);  // captured launches hold the old threshold
  c->gemv_max = max_tokens;
  return PW_OK;
}

// ================================================================== profiling
pw_status pw_set_profiling(pw_ctx *c, int on) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (on && c->prof_ev.empty()) {
    c->prof_ev.resize((size_t)c->d.L * 5, nullptr);
    for (auto &e : c->prof_ev) CU(c, cudaEventCreate(&e));
  }
  c->profiling = on ? 1 : 0;
  return PW_OK;
}

pw_status pw_profile_read(pw_ctx *c, int layer, float *ms) {
  if (!c || !ms) return fail(c, PW_ERR_INVALID, "null argument");
  if (layer < 0 || layer >= c->d.L) return fail(c, PW_ERR_INVALID, "layer out of range");
  if (c->prof_ev.empty()) return fail(c, PW_ERR_STATE, "profiling was never enabled");
  cudaEvent_t *e = &c->prof_ev[(size_t)layer * 5];
  CU(c, cudaEventSynchronize(e[4]));
  for (int k = 0; k < 4; ++k) CU(c, cudaEventElapsedTime(&ms[k], e[k], e[k + 1]));
  return PW_OK;
}

}  // extern "C"

// ================================================================== device-side timeouts
extern "C" pw_status pw_check(pw_ctx *c) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  CU(c, cudaStreamSynchronize(c->compute));
  int err = 0;
  CU(c, cudaMemcpy(&err, c->s.err, sizeof(int), cudaMemcpyDeviceToHost));
  if (err) {
    CU(c, cudaMemset(c->s.err, 0, sizeof(int)));
    if (err & pw::kErrWaitMask)
      return fail(c, PW_ERR_TIMEOUT, "a bounded device wait expired; that launch's outputs are invalid");
    return fail(c, PW_ERR_RANGE,
                "an activation left the fp16 range (|x| or |h| >= 65520, or NaN) or y is not finite; the outputs "
                "since the last check are invalid");
  }
  return check_sticky(c);
}

// ================================================================== helpers for pw_static.cu
namespace pw {

pw_status route_args(pw_ctx *c, int layer, const void *x, int T, int32_t *ids, float *w, int flags,
                     FwdArgs *a) {
  if (!c) return fail(nullptr, PW_ERR_INVALID, "null context");
  if (pw_status st = check_sticky(c)) return st;
  return forward_args(c, layer, x, T, const_cast<void *>(x), ids, w, flags, a);
}

pw_status report(pw_ctx *c, pw_status st, const char *msg) { return fail(c, st, "%s", msg); }

int ctx_device(const pw_ctx *c) { return c->d.device; }

}  // namespace pw
