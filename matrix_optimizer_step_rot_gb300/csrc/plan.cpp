// Host-side micro-group planner and the device memory layout it implies.
//
// Planner: Canzona page, section 3.2.2 "微组调度算法" -- sort every parameter
// by compute cost (descending), then grow micro-groups greedily: each item is
// tentatively added to the current group, a min-heap simulates which rank
// would take it, and if a byte cap is exceeded the addition is rolled back and
// a new group is opened.  Costs are m^2 n + m n^2 + m^3 + n^3 (the work of the
// two-sided rotation and the two bases), bytes are 4 m n (one float32 matrix).
#include "plan.h"

#include <algorithm>
#include <new>
#include <numeric>
#include <queue>

namespace rot {

uint64_t item_cost(int64_t m, int64_t n) {
  const uint64_t um = (uint64_t)m, un = (uint64_t)n;
  return um * um * un + um * un * un + um * um * um + un * un * un;
}

uint64_t item_bytes(int64_t m, int64_t n) { return 4ull * (uint64_t)m * (uint64_t)n; }

namespace {

// Heap entry: (accumulated cost, rank id); the top is the least loaded rank,
// ties broken towards the lowest id.
struct Load {
  uint64_t cost;
  int32_t rank;
};
struct MoreLoaded {
  bool operator()(const Load& a, const Load& b) const {
    return a.cost != b.cost ? a.cost > b.cost : a.rank > b.rank;
  }
};
using Heap = std::priority_queue<Load, hvec<Load>, MoreLoaded>;

Heap fresh_heap(int32_t ranks) {
  Heap h;
  for (int32_t r = 0; r < ranks; ++r) h.push({0, r});
  return h;
}

}  // namespace

void build_groups(rot_plan* p) {
  const int32_t count = p->count;
  hvec<uint64_t> cost(count), bytes(count);
  for (int32_t i = 0; i < count; ++i) {
    cost[i] = item_cost(p->shapes[i].m, p->shapes[i].n);
    bytes[i] = item_bytes(p->shapes[i].m, p->shapes[i].n);
  }
  hvec<int32_t> order(count);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return cost[a] > cost[b]; });

  p->owners.assign(count, -1);
  hvec<int32_t> current;
  Heap heap = fresh_heap(p->ranks);
  hvec<uint64_t> held(p->ranks, 0);  // bytes per rank in the current group
  uint64_t held_max = 0;

  auto close_group = [&]() {
    if (current.empty()) return;
    uint64_t b = 0, c = 0;
    for (int32_t i : current) b += bytes[i], c += cost[i];
    p->groups.push_back(current);
    p->group_bytes.push_back(b);
    p->group_cost.push_back(c);
    current.clear();
  };

  for (int32_t i : order) {
    Load top = heap.top();
    const uint64_t trial = held[top.rank] + bytes[i];
    if (!current.empty() && std::max(held_max, trial) > p->c_max) {
      // roll back: the item opens a new group with a fresh load simulation
      close_group();
      heap = fresh_heap(p->ranks);
      std::fill(held.begin(), held.end(), 0);
      held_max = 0;
      top = heap.top();
    }
    heap.pop();
    heap.push({top.cost + cost[i], top.rank});
    held[top.rank] += bytes[i];
    held_max = std::max(held_max, held[top.rank]);
    p->owners[i] = top.rank;
    current.push_back(i);
  }
  close_group();
}

// ---------------------------------------------------------------------------
// Device layout
// ---------------------------------------------------------------------------

namespace {

struct Cursor {
  uint64_t at = 0;
  hvec<uint64_t>* guards = nullptr;  // bounds-checked builds: a guard after every slice
  uint64_t take(uint64_t bytes) {
    const uint64_t o = at;
    at = align256(at + bytes);
    if (guards) {
      guards->push_back(at);
      at += kGuardBytes;
    }
    return o;
  }
  uint64_t floats(int64_t rows, int64_t ld) { return take(4ull * (uint64_t)rows * (uint64_t)ld); }
  uint64_t halves(int64_t rows, int64_t ld) { return take(2ull * (uint64_t)rows * (uint64_t)ld); }
};

}  // namespace

void build_layout(rot_plan* p) {
  Cursor s;
  const bool compact = p->state_format == ROT_STATE_COMPACT;
  s.take(256);                                   // status word (+ padding)
  p->ranks_off = s.take(8ull * (uint64_t)std::max(p->count, 1));
  p->zeros_off = 0;
  p->zeros_bytes = 0;
  if (compact) {  // one array of zeros as large as the largest basis
    int64_t most = 0;
    for (int32_t i = 0; i < p->count; ++i)
      for (int64_t d : {(int64_t)p->shapes[i].m, (int64_t)p->shapes[i].n})
        most = std::max(most, d * pad_ld(d));
    p->zeros_bytes = 2ull * (uint64_t)std::max<int64_t>(most, 1);
    p->zeros_off = s.take(p->zeros_bytes);
  }
  p->items.resize(p->count);
  for (int32_t i = 0; i < p->count; ++i) {
    ItemLayout& L = p->items[i];
    const int64_t m = p->shapes[i].m, n = p->shapes[i].n;
    L.m = (int)m;
    L.n = (int)n;
    L.ldm = (int)pad_ld(m);
    L.ldn = (int)pad_ld(n);
    if (compact) {
      L.mom = s.halves(m, L.ldn);
      L.v = s.floats(m, L.ldn);
      L.mt = s.halves(m, L.ldn);
      L.u16_hi = s.halves(m, L.ldm);
      L.ut16_hi = s.halves(m, L.ldm);
      L.vb16_hi = s.halves(n, L.ldn);
      L.vt16_hi = s.halves(n, L.ldn);
      continue;
    }
    L.mom = s.floats(m, L.ldn);
    L.v = s.floats(m, L.ldn);
    L.mt = s.floats(m, L.ldn);
    L.u16_hi = s.halves(m, L.ldm);
    L.u16_lo = s.halves(m, L.ldm);
    L.ut16_hi = s.halves(m, L.ldm);
    L.ut16_lo = s.halves(m, L.ldm);
    L.vb16_hi = s.halves(n, L.ldn);
    L.vb16_lo = s.halves(n, L.ldn);
    L.vt16_hi = s.halves(n, L.ldn);
    L.vt16_lo = s.halves(n, L.ldn);
  }
  if (compact)
    for (ItemLayout& L : p->items)
      L.u16_lo = L.ut16_lo = L.vb16_lo = L.vt16_lo = p->zeros_off;
  p->state_bytes = s.at;

  // Workspace: per group, a rotation region, the TF32 splits of the bases
  // and of M, then a refresh region.  The gradient split written by the
  // momentum kernel stays live across the refresh, so the regions do not
  // overlap.
  p->work.resize(p->groups.size());
  p->guards.assign(p->groups.size(), hvec<uint64_t>());
  uint64_t most = 256;
  for (size_t g = 0; g < p->groups.size(); ++g) {
    Cursor w;
    if (kChecked) w.guards = &p->guards[g];
    hvec<WorkLayout>& WL = p->work[g];
    WL.resize(p->groups[g].size());
    for (size_t k = 0; k < p->groups[g].size(); ++k) {
      const ItemLayout& L = p->items[p->groups[g][k]];
      WorkLayout& x = WL[k];
      x.g_hi = w.floats(L.m, L.ldn);
      x.g_lo = w.floats(L.m, L.ldn);
      x.sg_hi = w.floats(L.n, L.ldm);
      x.sg_lo = w.floats(L.n, L.ldm);
      x.sm_hi = w.floats(L.n, L.ldm);
      x.sm_lo = w.floats(L.n, L.ldm);
      x.gt = w.floats(L.m, L.ldn);
      x.mt = w.floats(L.m, L.ldn);
      x.g_rinv = w.floats(1, L.m);
      x.d_rinv = w.floats(1, L.m);
      x.m_rinv = w.floats(1, L.m);
      x.m16_hi = w.halves(L.m, L.ldn);
      x.m16_lo = w.halves(L.m, L.ldn);
    }
    {
      const uint64_t norms = w.floats(1, 4 * (int64_t)WL.size());
      for (size_t k = 0; k < WL.size(); ++k) {
        WL[k].g_rmax = norms + 16 * k;
        WL[k].d_rmax = norms + 16 * k + 4;
        WL[k].m_rmax = norms + 16 * k + 8;
        WL[k].m_amax = norms + 16 * k + 12;
      }
    }
    for (size_t k = 0; k < p->groups[g].size(); ++k) {
      const ItemLayout& L = p->items[p->groups[g][k]];
      WorkLayout& x = WL[k];
      x.u_hi = w.floats(L.m, L.ldm);
      x.u_lo = w.floats(L.m, L.ldm);
      x.ut_hi = w.floats(L.m, L.ldm);
      x.ut_lo = w.floats(L.m, L.ldm);
      x.vb_hi = w.floats(L.n, L.ldn);
      x.vb_lo = w.floats(L.n, L.ldn);
      x.vt_hi = w.floats(L.n, L.ldn);
      x.vt_lo = w.floats(L.n, L.ldn);
      x.m_hi = w.floats(L.m, L.ldn);
      x.m_lo = w.floats(L.m, L.ldn);
    }
    for (size_t k = 0; k < p->groups[g].size(); ++k) {
      const ItemLayout& L = p->items[p->groups[g][k]];
      WorkLayout& x = WL[k];
      x.mT_hi = w.floats(L.n, L.ldm);
      x.mT_lo = w.floats(L.n, L.ldm);
      // U side: Z_U^T = (M^T U)^T (m x n) when n < m, else Gram M M^T (m x m)
      const bool u_form1 = L.n < L.m;
      x.zu_rows = L.m;
      x.zu_ld = u_form1 ? L.ldn : L.ldm;
      x.zu_hi = w.floats(x.zu_rows, x.zu_ld);
      x.zu_lo = w.floats(x.zu_rows, x.zu_ld);
      // V side: Z_V^T = (M V)^T (n x m) when m < n, else Gram M^T M (n x n)
      const bool v_form1 = L.m < L.n;
      x.zv_rows = L.n;
      x.zv_ld = v_form1 ? L.ldm : L.ldn;
      x.zv_hi = w.floats(x.zv_rows, x.zv_ld);
      x.zv_lo = w.floats(x.zv_rows, x.zv_ld);
      x.aut_hi = w.floats(L.m, L.ldm);
      x.aut_lo = w.floats(L.m, L.ldm);
      x.avt_hi = w.floats(L.n, L.ldn);
      x.avt_lo = w.floats(L.n, L.ldn);
      x.qut_hi = w.floats(L.m, L.ldm);
      x.qut_lo = w.floats(L.m, L.ldm);
      x.qvt_hi = w.floats(L.n, L.ldn);
      x.qvt_lo = w.floats(L.n, L.ldn);
      const int rmax = std::min(L.m, L.n);
      x.aux_u = w.take(qr_aux_bytes(L.m, rmax));
      x.aux_v = w.take(qr_aux_bytes(L.n, rmax));
    }
    most = std::max(most, w.at);
  }
  p->work_bytes = most;
}

}  // namespace rot

// ---------------------------------------------------------------------------
// C ABI: plan
// ---------------------------------------------------------------------------

extern "C" {

int rot_plan_create_ex(const rot_shape* shapes, int32_t count, uint64_t c_max_bytes,
                       int32_t ranks, rot_plan** out) {
  if (!out) return ROT_EINVAL;
  *out = nullptr;
  if (count < 0 || (count > 0 && !shapes) || c_max_bytes == 0 || ranks < 1) return ROT_EINVAL;
  for (int32_t i = 0; i < count; ++i)
    if (shapes[i].m < 1 || shapes[i].n < 1 || shapes[i].m > ROT_MAX_DIM ||
        shapes[i].n > ROT_MAX_DIM)
      return ROT_EINVAL;
  rot_plan* p = new (std::nothrow) rot_plan();
  if (!p) return ROT_ENOMEM;
  try {
    p->count = count;
    p->ranks = ranks;
    p->c_max = c_max_bytes;
    p->shapes.assign(shapes, shapes + count);
    rot::build_groups(p);
    rot::build_layout(p);
  } catch (...) {
    delete p;
    return ROT_ENOMEM;
  }
  *out = p;
  return ROT_OK;
}

int rot_plan_create(const rot_shape* shapes, int32_t count, uint64_t c_max_bytes,
                    rot_plan** out) {
  return rot_plan_create_ex(shapes, count, c_max_bytes, 1, out);
}

void rot_plan_destroy(rot_plan* plan) { delete plan; }

int rot_plan_groups(const rot_plan* plan, int32_t* n_groups) {
  if (!plan || !n_groups) return ROT_EINVAL;
  *n_groups = (int32_t)plan->groups.size();
  return ROT_OK;
}

int rot_plan_group(const rot_plan* plan, int32_t g, const int32_t** items, int32_t* n_items,
                   uint64_t* bytes, uint64_t* cost) {
  if (!plan || g < 0 || g >= (int32_t)plan->groups.size()) return ROT_EINVAL;
  if (items) *items = plan->groups[g].data();
  if (n_items) *n_items = (int32_t)plan->groups[g].size();
  if (bytes) *bytes = plan->group_bytes[g];
  if (cost) *cost = plan->group_cost[g];
  return ROT_OK;
}

int rot_plan_owners(const rot_plan* plan, const int32_t** owners) {
  if (!plan || !owners) return ROT_EINVAL;
  *owners = plan->owners.data();
  return ROT_OK;
}

int rot_plan_set_state_format(rot_plan* plan, int32_t format) {
  if (!plan || (format != ROT_STATE_FULL && format != ROT_STATE_COMPACT)) return ROT_EINVAL;
  if (plan->state_format == format) return ROT_OK;
  try {
    plan->state_format = format;
    rot::build_layout(plan);
  } catch (const std::bad_alloc&) {
    return ROT_ENOMEM;
  }
  return ROT_OK;
}

int rot_state_bytes(const rot_plan* plan, uint64_t* state_bytes, uint64_t* work_bytes) {
  if (!plan) return ROT_EINVAL;
  if (state_bytes) *state_bytes = plan->state_bytes;
  if (work_bytes) *work_bytes = plan->work_bytes;
  return ROT_OK;
}

}  // extern "C"
