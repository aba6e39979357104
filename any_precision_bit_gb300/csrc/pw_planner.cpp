// pw_planner.cpp -- the quality-aware runtime planner of PagedWeight Sec. 3.2 (Algorithm 1,
// PlanStep), host only.
//
//   D       = max{0, T_blk + 1 - F_blk} * B_KV                           (Eq. 7)
//   g       = max{s^{b'} - s^b, 0}                                       (Eq. 4)
//   rho_hat = w_u^{b->b'} . phi_i + a_u^{b->b'}                          (Eq. 5)
//             (or read from a batch-level table, obs->rho_hat)
//   eta     = exp(alpha * c_u^{b->b'} * clip(rho_hat, rho_min, rho_max)) (Eq. 6)
//   d_hat   = max{eps, mu_beta * g * eta}                                (Eq. 8)
//   Delta   = M^b - M^{b'}                                               (Eq. 3)
//
// A step is one level b -> b' (the next lower supported bitwidth); taking a block's step
// unlocks its next one.  Each bitwidth-floor stage s allows blocks to end at most s+1
// levels below their committed bitwidth and never below their bucket's floor; its greedy
// pass takes the smallest d_hat / Delta first (ties: larger Delta, then lower block) until
// D bytes are released.  Under pressure (D > 0) the lowest stage meeting D is chosen,
// else the stage releasing the most bytes.  Buckets come from routing mass (Eq. 1): the
// experts of a layer sorted by mass (ties to the lower id), rank r -> bucket
// r * n_buckets / E, bucket 0 hottest.  With no pressure and F_blk >= T_blk + R a reload
// plan restores single levels toward the initial bitwidths, largest d_hat / Delta first,
// while the restored bytes fit in (F_blk - T_blk - R) * B_KV.
#include <algorithm>
#include <cmath>
#include <queue>
#include <vector>

#include "../../include/pw.h"

namespace {

struct Step {
  double key, delta;
  int block;
};

struct Ctx {
  const pw_plan_problem *p;
  const pw_obs *o;
  const pw_offline *f;
  std::vector<int> beta;   // bucket per block
  std::vector<int> level;  // committed level per block
  std::vector<int> top;    // initial level per block
};

int level_of(const pw_plan_problem *p, int b) {
  for (int j = 0; j < p->n_bits; ++j)
    if (p->bits[j] == b) return j;
  return -1;
}

// d_hat and Delta of block i going from level j to level j-1
void score(const Ctx &c, int i, int j, double *d_hat, double *delta) {
  const pw_plan_problem *p = c.p;
  const pw_offline *f = c.f;
  const int nb = p->n_bits, u = p->utype[i], tr = j - 1;
  const double s_hi = f->s[(size_t)i * nb + j], s_lo = f->s[(size_t)i * nb + j - 1];
  const double g = std::max(s_lo - s_hi, 0.0);
  double rho = 0.0;
  if (c.o->rho_hat) {
    rho = c.o->rho_hat[(size_t)i * (nb - 1) + tr];
  } else {
    const double *w = f->head_w + ((size_t)u * (nb - 1) + tr) * 3;
    const double *phi = c.o->phi + (size_t)i * 3;
    for (int m = 0; m < 3; ++m) rho = rho + w[m] * phi[m];
    rho = rho + f->head_a[(size_t)u * (nb - 1) + tr];
  }
  const double cl = std::min(std::max(rho, f->rho_min), f->rho_max);
  const double eta = std::exp(f->alpha * f->head_c[(size_t)u * (nb - 1) + tr] * cl);
  *d_hat = std::max(f->eps, f->mu[c.beta[i]] * g * eta);
  *delta = p->M[(size_t)i * nb + j] - p->M[(size_t)i * nb + j - 1];
}

struct Cheaper {  // priority_queue puts the "largest" first: invert for min-heap order
  bool operator()(const Step &a, const Step &b) const {
    if (a.key != b.key) return a.key > b.key;
    if (a.delta != b.delta) return a.delta < b.delta;
    return a.block > b.block;
  }
};

struct Costlier {
  bool operator()(const Step &a, const Step &b) const {
    if (a.key != b.key) return a.key < b.key;
    if (a.delta != b.delta) return a.delta < b.delta;
    return a.block > b.block;
  }
};

struct StagePlan {
  std::vector<int> to_level;  // -1 untouched
  std::vector<double> released;
  double total = 0.0;
};

StagePlan greedy(const Ctx &c, int cap, double D) {
  const int n = c.p->n_blocks;
  StagePlan sp;
  sp.to_level.assign(n, -1);
  sp.released.assign(n, 0.0);
  if (D <= 0) return sp;
  std::vector<int> cur = c.level;
  std::priority_queue<Step, std::vector<Step>, Cheaper> heap;
  auto push = [&](int i) {
    const int j = cur[i];
    if (j == 0) return;
    if (c.p->bits[j - 1] < c.f->floors[c.beta[i]]) return;
    if (c.level[i] - (j - 1) > cap) return;
    double d_hat, delta;
    score(c, i, j, &d_hat, &delta);
    heap.push(Step{d_hat / delta, delta, i});
  };
  for (int i = 0; i < n; ++i) push(i);
  while (!heap.empty() && sp.total < D) {
    Step s = heap.top();
    heap.pop();
    cur[s.block] -= 1;
    sp.total += s.delta;
    sp.released[s.block] += s.delta;
    sp.to_level[s.block] = cur[s.block];
    push(s.block);
  }
  return sp;
}

StagePlan reload(const Ctx &c, double budget) {
  const int n = c.p->n_blocks;
  StagePlan sp;
  sp.to_level.assign(n, -1);
  sp.released.assign(n, 0.0);
  std::vector<int> cur = c.level;
  std::priority_queue<Step, std::vector<Step>, Costlier> heap;
  auto push = [&](int i) {
    const int j = cur[i];
    if (j >= c.top[i]) return;
    double d_hat, delta;
    score(c, i, j + 1, &d_hat, &delta);
    heap.push(Step{d_hat / delta, delta, i});
  };
  for (int i = 0; i < n; ++i) push(i);
  while (!heap.empty()) {
    Step s = heap.top();
    if (sp.total + s.delta > budget) break;
    heap.pop();
    cur[s.block] += 1;
    sp.total += s.delta;
    sp.released[s.block] += s.delta;
    sp.to_level[s.block] = cur[s.block];
    push(s.block);
  }
  return sp;
}

pw_status emit(const Ctx &c, const StagePlan &sp, int kind, int stage, double D, pw_plan *out) {
  out->kind = kind;
  out->stage = stage;
  out->D = D;
  out->total = sp.total;
  out->n = 0;
  for (int i = 0; i < c.p->n_blocks; ++i) {
    if (sp.to_level[i] < 0) continue;
    if (out->n >= out->capacity) return PW_ERR_INVALID;
    pw_plan_entry &e = out->entries[out->n++];
    e.block = i;
    e.from_bits = c.p->bits[c.level[i]];
    e.to_bits = c.p->bits[sp.to_level[i]];
    e.delta = sp.released[i];
  }
  return PW_OK;
}

}  // namespace

extern "C" pw_status pw_plan_host(const pw_plan_problem *p, const pw_obs *o, const pw_offline *f, pw_plan *out) {
  if (!p || !o || !f || !out || (!out->entries && out->capacity > 0)) return PW_ERR_INVALID;
  if (p->n_blocks < 0 || p->n_bits < 1 || p->n_bits != f->n_bits || p->L < 1 || p->E < 1) return PW_ERR_INVALID;
  if (!p->bits || !p->q || !p->utype || !p->layer || !p->expert || !p->M || !(o->phi || o->rho_hat) || !o->mass)
    return PW_ERR_INVALID;
  if (!f->s || !f->head_w || !f->head_a || !f->head_c || !f->mu || !f->floors) return PW_ERR_INVALID;
  if (f->n_buckets < 1 || f->n_stages < 1) return PW_ERR_INVALID;
  Ctx c{p, o, f, {}, {}, {}};
  const int n = p->n_blocks;
  c.level.resize(n);
  c.top.resize(n);
  c.beta.resize(n);
  for (int i = 0; i < n; ++i) {
    c.level[i] = level_of(p, p->q[i]);
    c.top[i] = p->q_init ? level_of(p, p->q_init[i]) : c.level[i];
    if (c.level[i] < 0 || c.top[i] < 0) return PW_ERR_INVALID;
    if (p->layer[i] < 0 || p->layer[i] >= p->L || p->expert[i] < 0 || p->expert[i] >= p->E) return PW_ERR_INVALID;
    if (p->utype[i] != 0 && p->utype[i] != 1) return PW_ERR_INVALID;
  }
  // buckets from routing mass, per layer
  std::vector<int> bucket((size_t)p->L * p->E);
  std::vector<int> order(p->E);
  for (int l = 0; l < p->L; ++l) {
    for (int e = 0; e < p->E; ++e) order[e] = e;
    const double *m = o->mass + (size_t)l * p->E;
    std::sort(order.begin(), order.end(), [m](int a, int b) {
      if (m[a] != m[b]) return m[a] > m[b];
      return a < b;
    });
    for (int r = 0; r < p->E; ++r) bucket[(size_t)l * p->E + order[r]] = (int)(((long)r * f->n_buckets) / p->E);
  }
  for (int i = 0; i < n; ++i) c.beta[i] = bucket[(size_t)p->layer[i] * p->E + p->expert[i]];

  const double D = std::max(0, o->T_blk + 1 - o->F_blk) * o->B_KV;
  std::vector<StagePlan> queue;
  for (int s = 0; s < f->n_stages; ++s) queue.push_back(greedy(c, s + 1, D));
  if (D > 0) {
    int pick = -1;
    for (int s = 0; s < f->n_stages && pick < 0; ++s)
      if (queue[s].total >= D) pick = s;
    if (pick < 0) {
      pick = 0;
      for (int s = 1; s < f->n_stages; ++s)
        if (queue[s].total > queue[pick].total) pick = s;
    }
    return emit(c, queue[pick], 1, pick, D, out);
  }
  if (o->F_blk >= o->T_blk + o->R) {
    StagePlan r = reload(c, (double)(o->F_blk - o->T_blk - o->R) * o->B_KV);
    return emit(c, r, r.total > 0 ? 2 : 0, -1, D, out);
  }
  StagePlan none;
  none.to_level.assign(n, -1);
  none.released.assign(n, 0.0);
  return emit(c, none, 0, -1, D, out);
}

extern "C" pw_status pw_merge_requests(const pw_request_signals *req, int n_req, int L, int E, int n_blocks,
                                       int n_bits, double *mass, double *rho_hat, double *conf, double *rho_min,
                                       double *rho_max) {
  if (!req || n_req < 1 || L < 1 || E < 1 || n_blocks < 0 || n_bits < 1) return PW_ERR_INVALID;
  if (!mass || !rho_hat || !conf || !rho_min || !rho_max) return PW_ERR_INVALID;
  double tot = 0.0;
  for (int r = 0; r < n_req; ++r) {
    if (!req[r].mass || !req[r].rho_hat || !req[r].conf || !(req[r].kv_blocks >= 0.0)) return PW_ERR_INVALID;
    tot += req[r].kv_blocks;
  }
  if (!(tot > 0.0)) return PW_ERR_INVALID;
  const size_t nm = (size_t)L * E, nr = (size_t)n_blocks * (n_bits - 1), nc = (size_t)2 * (n_bits - 1);
  for (size_t i = 0; i < nm; ++i) mass[i] = 0.0;
  for (size_t i = 0; i < nr; ++i) rho_hat[i] = 0.0;
  for (size_t i = 0; i < nc; ++i) conf[i] = 0.0;
  *rho_min = 0.0;
  *rho_max = 0.0;
  for (int r = 0; r < n_req; ++r) {
    const double w = req[r].kv_blocks / tot;
    for (size_t i = 0; i < nm; ++i) mass[i] = mass[i] + w * req[r].mass[i];
    for (size_t i = 0; i < nr; ++i) rho_hat[i] = rho_hat[i] + w * req[r].rho_hat[i];
    for (size_t i = 0; i < nc; ++i) conf[i] = conf[i] + w * req[r].conf[i];
    *rho_min = *rho_min + w * req[r].rho_min;
    *rho_max = *rho_max + w * req[r].rho_max;
  }
  return PW_OK;
}
