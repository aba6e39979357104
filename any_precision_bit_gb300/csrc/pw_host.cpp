// pw_host.cpp -- host-only pieces of the ABI: the plain bit-plane packer, the kernel-private
// plane tiling and its inverse, and the context-level planner entry point.
#include <cuda_runtime.h>

#include <cstring>
#include <vector>

#include "../../include/pw.h"
#include "pw_internal.h"

using namespace pw;

extern "C" {

// Plain layout: plane p holds bit (bmax-1-p) of every code (PagedWeight Sec. 2.2: a b-bit
// code is the top b planes); bit j of word w of a plane row is column 32w + j.
pw_status pw_pack_planes_host(const uint8_t *idx, int N, int K, int bmax, uint32_t *planes) {
  if (!idx || !planes || N < 1 || K < 1 || bmax < 1 || bmax > 8) return PW_ERR_INVALID;
  const int W = kpad_cols(K) / 32;
  std::memset(planes, 0, sizeof(uint32_t) * (size_t)bmax * N * W);
  for (int n = 0; n < N; ++n) {
    const uint8_t *row = idx + (size_t)n * K;
    for (int k = 0; k < K; ++k) {
      const unsigned code = row[k];
      if (code >> bmax) return PW_ERR_INVALID;
      for (int p = 0; p < bmax; ++p)
        planes[((size_t)p * N + n) * W + k / 32] |= ((code >> (bmax - 1 - p)) & 1u) << (k % 32);
    }
  }
  return PW_OK;
}

static bool tile_args_ok(const uint32_t *a, const uint32_t *b, int N, int K, int nplanes, int u) {
  return a && b && N >= 16 && N % 16 == 0 && K >= 1 && nplanes >= 1 && nplanes <= 8 && (u == 0 || u == 1);
}

pw_status pw_tile_planes_host(const uint32_t *planes, int N, int K, int nplanes, int u, uint32_t *tiled) {
  if (!tile_args_ok(planes, tiled, N, K, nplanes, u)) return PW_ERR_INVALID;
  const int Kp = kpad_cols(K), W = Kp / 32, KC = Kp / kChunkCols, I = N / 2;
  const size_t per = (size_t)N * W;
  std::memset(tiled, 0, sizeof(uint32_t) * per * nplanes);
  for (int p = 0; p < nplanes; ++p)
    for (int d = 0; d < N; ++d) {
      const int r = orig_row(d, u, I);
      for (int k = 0; k < Kp; ++k) {
        const uint32_t bit = (planes[p * per + (size_t)r * W + k / 32] >> (k % 32)) & 1u;
        long word;
        int pos;
        tile_pos(d, k, N, KC, &word, &pos);
        tiled[p * per + word] |= bit << pos;
      }
    }
  return PW_OK;
}

pw_status pw_untile_planes_host(const uint32_t *tiled, int N, int K, int nplanes, int u, uint32_t *planes) {
  if (!tile_args_ok(tiled, planes, N, K, nplanes, u)) return PW_ERR_INVALID;
  const int Kp = kpad_cols(K), W = Kp / 32, KC = Kp / kChunkCols, I = N / 2;
  const size_t per = (size_t)N * W;
  std::memset(planes, 0, sizeof(uint32_t) * per * nplanes);
  for (int p = 0; p < nplanes; ++p)
    for (int d = 0; d < N; ++d) {
      const int r = orig_row(d, u, I);
      for (int k = 0; k < Kp; ++k) {
        long word;
        int pos;
        tile_pos(d, k, N, KC, &word, &pos);
        const uint32_t bit = (tiled[p * per + word] >> pos) & 1u;
        planes[p * per + (size_t)r * W + k / 32] |= bit << (k % 32);
      }
    }
  return PW_OK;
}

}  // extern "C"
