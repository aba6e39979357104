// Host check of the expert kernels' work lists (compiled and run by test_worklist_host.py).
//
// The router writes per-projection tables (the first item of each expert rank, the expert
// at each rank) and work_item() expands item i from them.  For random layer shapes, routing
// counts and bitwidths this checks what the lists must satisfy, without restating how
// work_item() computes an item:
//   * shared-expert items come first; every (row tile, token chunk) of the shared expert,
//     and for the down projection every K part of it, appears exactly once; the parts of a
//     (tile, chunk) are non-empty and tile [0, stages) in order;
//   * every (row tile, slot chunk) of every expert with routed tokens appears exactly once,
//     and for the down projection every K part of it (one part for prefill-sized batches);
//     the parts are non-empty and tile the expert's K in order; an expert's items are
//     contiguous, and the experts come by decreasing bitwidth, ties by expert id; experts
//     without tokens have no items;
//   * token ranges are within the batch (shared) or the expert's slots (routed), and each
//     chunk except an expert's or the batch's last holds tok_chunk_for(T) tokens;
//   * the shared items the expert kernels build by themselves, from their count alone (they
//     start before the tables exist), are the list's.
// Exit status 0 when every check passes; the first failure is printed.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <tuple>
#include <vector>

#include "pw_internal.h"

using namespace pw;

static int fail(const char *what, int trial, int u, int i) {
  std::printf("FAIL %s (trial %d, projection %d, item %d)\n", what, trial, u, i);
  return 1;
}

static unsigned rng_state = 12345u;
static int rnd(int n) {  // uniform in [0, n)
  rng_state = rng_state * 1664525u + 1013904223u;
  return (int)((rng_state >> 8) % (unsigned)n);
}

int main() {
  for (int trial = 0; trial < 400; ++trial) {
    const int E = 1 + rnd(256);
    const int K = 1 + rnd(E < 8 ? E : 8);
    const int T = 1 + (rnd(3) == 0 ? rnd(4096) : rnd(300));
    const int H = 16 * (1 + rnd(300));
    // one routed down stage, long routed downs (many K parts at decode sizes), or in between
    const int I = 16 * (1 + rnd(trial % 4 == 0 ? 8 : (trial % 4 == 1 ? 1024 : 200)));
    const int Is = rnd(2) ? 16 * (1 + rnd(600)) : 0;
    std::vector<int> cnt(E, 0), q(E), q2(E);
    for (int t = 0; t < T; ++t) {  // K distinct experts per token
      std::vector<int> ids(E);
      for (int e = 0; e < E; ++e) ids[e] = e;
      for (int k = 0; k < K; ++k) {
        const int j = k + rnd(E - k);
        const int tmp = ids[k];
        ids[k] = ids[j];
        ids[j] = tmp;
        ++cnt[ids[k]];
      }
    }
    for (int e = 0; e < E; ++e) {
      q[e] = 3 + rnd(6);
      q2[e] = 3 + rnd(6);
    }
    const int tc = tok_chunk_for(T), tchunks = (T + tc - 1) / tc;
    const int tiles[2] = {(2 * I + kCtaRows - 1) / kCtaRows, (H + kCtaRows - 1) / kCtaRows};
    const int sh_tiles[2] = {(2 * Is + kCtaRows - 1) / kCtaRows, (H + kCtaRows - 1) / kCtaRows};
    const int nsplit = shared_down_splits(I, Is);
    const int stages = (Is / 16 + 7) / 8;
    const int kc_full[2] = {kpad_cols(H) / kChunkCols, kpad_cols(I) / kChunkCols};
    if (nsplit < 1 || nsplit > 8) return fail("split count outside 1..8", trial, 1, -1);
    const int dsplit = routed_down_splits(T, I);
    if (dsplit < 1 || dsplit > 8 || (T >= kPrefillMinT && dsplit != 1)) return fail("routed split count", trial, 1, -1);
    std::vector<int> off(E + 1, 0);
    for (int e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
    for (int u = 0; u < 2; ++u) {
      const std::vector<int> &qu = u ? q2 : q;
      // the tables as the router lays them out: ranks by decreasing bitwidth, ties by id
      std::vector<int> rk(E), first(E + 1);
      for (int e = 0; e < E; ++e) {
        int r = 0;
        for (int f = 0; f < E; ++f) r += qu[f] > qu[e] || (qu[f] == qu[e] && f < e);
        rk[r] = e;
      }
      const int n_sh = Is > 0 ? sh_tiles[u] * tchunks * (u ? nsplit : 1) : 0;
      // the expert kernels count the shared items, and build them, without the tables
      if (shared_item_count(u, T, H, I, Is) != n_sh) return fail("shared item count", trial, u, -1);
      first[0] = n_sh;
      const int np = u ? dsplit : 1;
      for (int r = 0; r < E; ++r) first[r + 1] = first[r] + tiles[u] * np * ((cnt[rk[r]] + tc - 1) / tc);
      std::map<std::tuple<int, int, int>, int> seen_sh;            // (tile, chunk, part)
      std::map<std::tuple<int, int, int, int>, int> seen_rt;       // (expert, tile, chunk, part)
      std::map<std::tuple<int, int, int>, std::vector<std::pair<int, int>>> rparts;  // (expert, tile, chunk) -> kc ranges
      std::map<std::pair<int, int>, std::vector<std::pair<int, int>>> parts;  // (tile, chunk) -> kc ranges
      int prev_e = -1;
      std::vector<int> done(E, 0);
      for (int i = 0; i < first[E]; ++i) {
        const WorkItem w = work_item(u, i, first.data(), rk.data(), off.data(), E, T, H, I, Is);
        if (w.kc0 >= w.kc1) return fail("empty K range", trial, u, i);
        if (w.ntok < 1 || w.ntok > tc) return fail("token count", trial, u, i);
        if (i < n_sh) {
          if (w.kind != 1) return fail("shared items first", trial, u, i);
          const WorkItem wl = work_item(u, i, &n_sh, nullptr, nullptr, E, T, H, I, Is);
          if (wl.kind != w.kind || wl.tile != w.tile || wl.tok0 != w.tok0 || wl.ntok != w.ntok || wl.kc0 != w.kc0 ||
              wl.kc1 != w.kc1 || wl.part != w.part)
            return fail("shared item built without the tables differs", trial, u, i);
          if (w.tile < 0 || w.tile >= sh_tiles[u] || w.tok0 % tc || w.tok0 / tc >= tchunks)
            return fail("shared tile or chunk", trial, u, i);
          if (w.tok0 + w.ntok > T || (w.tok0 + w.ntok < T && w.ntok != tc)) return fail("shared tokens", trial, u, i);
          if (u == 0 && (w.kc0 != 0 || w.kc1 != kc_full[0])) return fail("shared gate_up K range", trial, u, i);
          if (u == 1 && (w.part < 0 || w.part >= nsplit)) return fail("shared part", trial, u, i);
          if (seen_sh[std::make_tuple(w.tile, w.tok0 / tc, w.part)]++) return fail("shared item twice", trial, u, i);
          if (u == 1) parts[std::make_pair(w.tile, w.tok0 / tc)].push_back(std::make_pair(w.kc0, w.kc1));
          continue;
        }
        if (w.kind != 0 || w.expert < 0 || w.expert >= E) return fail("routed expert", trial, u, i);
        const int e = w.expert;
        if (cnt[e] == 0) return fail("item of an expert without tokens", trial, u, i);
        if (e != prev_e) {
          if (done[e]) return fail("expert items not contiguous", trial, u, i);
          if (prev_e >= 0 && (qu[prev_e] < qu[e] || (qu[prev_e] == qu[e] && prev_e > e)))
            return fail("experts out of bitwidth order", trial, u, i);
          if (prev_e >= 0) done[prev_e] = 1;
          prev_e = e;
        }
        if (w.tile < 0 || w.tile >= tiles[u] || w.tok0 % tc) return fail("routed tile or chunk", trial, u, i);
        if (w.tok0 + w.ntok > cnt[e] || (w.tok0 + w.ntok < cnt[e] && w.ntok != tc)) return fail("routed tokens", trial, u, i);
        if (w.part < 0 || w.part >= np) return fail("routed part", trial, u, i);
        if (seen_rt[std::make_tuple(e, w.tile, w.tok0 / tc, w.part)]++) return fail("routed item twice", trial, u, i);
        rparts[std::make_tuple(e, w.tile, w.tok0 / tc)].push_back(std::make_pair(w.part, w.kc0 * 4096 + w.kc1));
      }
      // completeness
      if (Is > 0 && (int)seen_sh.size() != n_sh) return fail("shared items missing", trial, u, -1);
      long want = 0;
      for (int e = 0; e < E; ++e) want += (long)tiles[u] * np * ((cnt[e] + tc - 1) / tc);
      if ((long)seen_rt.size() != want) return fail("routed items missing", trial, u, -1);
      for (auto &kv : rparts) {  // the parts of an (expert, tile, chunk) tile its K in order
        auto v = kv.second;
        std::sort(v.begin(), v.end());
        int at = 0;
        for (auto &pr : v) {
          const int kc0 = pr.second / 4096, kc1 = pr.second % 4096;
          if (kc0 != at) return fail("routed parts not contiguous", trial, u, -1);
          at = kc1;
        }
        if (at != kc_full[u]) return fail("routed parts do not cover K", trial, u, -1);
      }
      for (auto &kv : parts) {  // the parts of a (tile, chunk) tile the shared down's K in order
        auto &v = kv.second;
        if ((int)v.size() != nsplit) return fail("part count", trial, u, -1);
        int at = 0;
        for (int p = 0; p < nsplit; ++p) {
          if (v[p].first != at) return fail("parts not contiguous", trial, u, -1);
          at = v[p].second;
        }
        if (at != stages) return fail("parts do not cover K", trial, u, -1);
      }
    }
  }
  std::printf("ok\n");
  return 0;
}
