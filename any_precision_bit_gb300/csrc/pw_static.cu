// pw_static.cu -- pw_route_noalloc: the routing kernel run on scratch that lives in a static
// device array of this library, so that the call allocates no memory.
//
// Who needs it: code that must not call cudaMalloc (or any allocating routine) at the point
// where it routes tokens -- for example a caller that runs under an external memory
// budget or allocator it does not control, or a host thread that may not touch the CUDA
// allocator while other work is in flight.  pw_moe_forward's own scratch is allocated by
// pw_create; this entry point uses none of it.
//
// The array below is part of the module: every GPU that loads libpw.so holds it until the
// process exits.  All calls share it and it keeps the last call's contents.
#include <cuda_runtime.h>

#include <cstdio>

#include "pw_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

// Host-side stand-in of g_route_scratch is not a device address: the real address is looked
// up once per device, with that device current.
void *g_scratch_addr[kMaxDevices] = {};

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace

extern "C" pw_status pw_route_noalloc(pw_ctx *ctx, int layer, const void *x, int T, int32_t *ids,
                                      float *w, int flags, pw_stream stream) {
  using namespace pw;
  if (!ctx || !ids || !w) return report(ctx, PW_ERR_INVALID, "pw_route_noalloc: null context, ids or w");
  const int dev = ctx_device(ctx);
  if (dev < 0 || dev >= kMaxDevices) return report(ctx, PW_ERR_INVALID, "pw_route_noalloc: device ordinal too large");
  FwdArgs a;
  if (pw_status st = route_args(ctx, layer, x, T, ids, w, flags & PW_PRENORM, &a)) return st;

  // scratch the router kernel touches, carved from the static array (256-byte aligned)
  // (the work items themselves are written from the rank tables by the gather kernel of a
  // forward, which this call does not run)
  const long TK = (long)T * a.K;
  const size_t sizes[] = {
      sizeof(float) * T * a.E,      // logits
      sizeof(int) * TK,             // ids
      sizeof(float) * TK,           // w
      sizeof(int) * 4 * kRankStride,  // ranks: the work-list tables
      sizeof(int) * (a.E + 1),      // offsets
      sizeof(int) * TK,             // slot_tok
      sizeof(int) * TK,             // pair_slot
      sizeof(float) * TK,           // slot_w
      0,                            // items1 (not used)
      0,                            // items2 (not used)
      sizeof(int) * 2,              // n_items
      sizeof(unsigned) * (1 + (T + 7) / 8),  // tickets: all token groups, then one per group
      sizeof(float) * T,            // inv_rms
      0,                            // stat_count (the router does not add statistics)
      0,                            // stat_wsum
      sizeof(uint16_t) * T * a.H,   // xh: the fp16 expert input the router also writes
      sizeof(float) * T,            // xnorm: per-token input norms
      sizeof(float) * T,            // sgate: per-token shared-expert gates (gated layers)
  };
  size_t need = 0;
  for (size_t s : sizes) need += align256(s);
  if (need > kStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof msg, "pw_route_noalloc: T=%d needs %zu bytes of scratch, the static array holds %zu",
             T, need, kStaticScratchBytes);
    return report(ctx, PW_ERR_INVALID, msg);
  }

  // one-time set-up per device, with that device current
  if (!g_scratch_addr[dev]) {
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(dev);
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    cudaSetDevice(prev);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return report(ctx, PW_ERR_CUDA, "pw_route_noalloc: cudaGetSymbolAddress failed");
    }
    g_scratch_addr[dev] = p;
  }
  char *base = static_cast<char *>(g_scratch_addr[dev]);
  char *cur = base;
  auto take = [&](size_t n) {
    char *p = cur;
    cur += align256(n);
    return p;
  };
  Scratch s{};
  s.logits = reinterpret_cast<float *>(take(sizes[0]));
  s.ids = reinterpret_cast<int *>(take(sizes[1]));
  s.w = reinterpret_cast<float *>(take(sizes[2]));
  s.ranks = reinterpret_cast<int *>(take(sizes[3]));
  s.offsets = reinterpret_cast<int *>(take(sizes[4]));
  s.slot_tok = reinterpret_cast<int *>(take(sizes[5]));
  s.pair_slot = reinterpret_cast<int *>(take(sizes[6]));
  s.slot_w = reinterpret_cast<float *>(take(sizes[7]));
  s.items1 = nullptr;
  s.items2 = nullptr;
  s.n_items = reinterpret_cast<int *>(take(sizes[10]));
  s.ticket = reinterpret_cast<unsigned *>(take(sizes[11]));
  s.inv_rms = reinterpret_cast<float *>(take(sizes[12]));
  s.stat_count = nullptr;  // the routing statistics are added by the forward's gather kernel
  s.stat_wsum = nullptr;
  s.xh = reinterpret_cast<uint16_t *>(take(sizes[15]));
  s.xnorm = reinterpret_cast<float *>(take(sizes[16]));
  s.sgate = reinterpret_cast<float *>(take(sizes[17]));
  s.max_items1 = 0;
  s.max_items2 = 0;
  // a router whose bounded wait for its copies expires records it in the context's own error
  // word (allocated by pw_create), which the next pw_check on the context reports
  s.err = a.s.err;
  a.s = s;  // a.layer still selects the layer's router, bias and page-table bitwidths

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the last-CTA tickets must start at zero; the array keeps whatever the last call left
  if (cudaMemsetAsync(s.ticket, 0, sizes[11], st) != cudaSuccess) {
    cudaGetLastError();
    return report(ctx, PW_ERR_CUDA, "pw_route_noalloc: clearing the ticket failed");
  }
  if (int e = launch_route(a, stream)) {
    char msg[160];
    snprintf(msg, sizeof msg, "pw_route_noalloc: launch failed: %s", cudaGetErrorString((cudaError_t)e));
    return report(ctx, PW_ERR_CUDA, msg);
  }
  return PW_OK;
}
