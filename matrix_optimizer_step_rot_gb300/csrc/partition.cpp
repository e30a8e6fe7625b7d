// Data-parallel partition of matrices over ranks (host only).
//
// Canzona page, section 3.1.1: static ownership by parameter start within a
// ZeRO-1 bucket.  Section 3.2.1: the alpha-balanced greedy LPT partition --
// buckets by work, largest first; per-rank deficits against the ideal load;
// shares mixed between an even split (alpha -> 0) and deficit filling
// (alpha -> 1); cuts placed on parameter boundaries.  The ideal load is the
// mean load before the bucket, sum L / R, as the page's code prints it
// (ROT_ALPHA_IDEAL_BEFORE), or, as an option, the even share once the bucket
// is placed, (sum L + W_b) / R (ROT_ALPHA_IDEAL_AFTER).
//
// The cuts are decided in float64.  This file is compiled without
// floating-point contraction, and every sum runs in a fixed order, so the
// cuts are the same on every host.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <new>
#include <numeric>
#include <vector>

#include "plan.h"
#include "rot.h"

using rot::hvec;

namespace {

constexpr uint64_t kExactLimit = 1ull << 53;  // integers exact in a double

// Checks the bucket sizes against `count`; fills the start index of each.
bool bucket_starts(const int32_t* sizes, int32_t n_buckets, int32_t count,
                   hvec<int64_t>& start) {
  start.resize((size_t)n_buckets);
  int64_t at = 0;
  for (int32_t b = 0; b < n_buckets; ++b) {
    if (sizes[b] < 0) return false;
    start[(size_t)b] = at;
    at += sizes[b];
  }
  return at == count;
}

bool bad_common(int32_t count, const int32_t* sizes, int32_t n_buckets, int32_t ranks,
                const void* in, const int32_t* owners) {
  if (count < 0 || n_buckets < 0 || ranks < 1) return true;
  if (count > 0 && (!in || !owners)) return true;
  if (n_buckets > 0 && !sizes) return true;
  return false;
}

}  // namespace

extern "C" int rot_item_work(const rot_shape* shapes, int32_t count, uint64_t* work) {
  if (count < 0 || (count > 0 && (!shapes || !work))) return ROT_EINVAL;
  for (int32_t i = 0; i < count; ++i) {
    const int32_t m = shapes[i].m, n = shapes[i].n;
    if (m < 1 || n < 1 || m > ROT_MAX_DIM || n > ROT_MAX_DIM) return ROT_EINVAL;
  }
  for (int32_t i = 0; i < count; ++i) work[i] = rot::item_cost(shapes[i].m, shapes[i].n);
  return ROT_OK;
}

extern "C" int rot_partition_static(const uint64_t* elems, int32_t count,
                                    const int32_t* bucket_sizes, int32_t n_buckets,
                                    int32_t ranks, int32_t* owners) {
  if (bad_common(count, bucket_sizes, n_buckets, ranks, elems, owners)) return ROT_EINVAL;
  try {
    hvec<int64_t> start;
    if (!bucket_starts(bucket_sizes, n_buckets, count, start)) return ROT_EINVAL;
    for (int32_t b = 0; b < n_buckets; ++b) {
      const int64_t s0 = start[(size_t)b], s1 = s0 + bucket_sizes[b];
      uint64_t total = 0;
      for (int64_t i = s0; i < s1; ++i) {
        if (elems[i] > UINT64_MAX - total) return ROT_EINVAL;
        total += elems[i];
      }
      const uint64_t R = (uint64_t)ranks;
      uint64_t shard = total / R + (total % R != 0 ? 1u : 0u);
      if (shard == 0) shard = 1;
      uint64_t offset = 0;
      for (int64_t i = s0; i < s1; ++i) {
        owners[i] = (int32_t)std::min<uint64_t>(R - 1, offset / shard);
        offset += elems[i];
      }
    }
  } catch (const std::bad_alloc&) {
    return ROT_ENOMEM;
  }
  return ROT_OK;
}

extern "C" int rot_partition_alpha_ex(const uint64_t* work, int32_t count,
                                      const int32_t* bucket_sizes, int32_t n_buckets,
                                      int32_t ranks, double alpha, int32_t ideal,
                                      int32_t* owners, uint64_t* loads) {
  if (bad_common(count, bucket_sizes, n_buckets, ranks, work, owners)) return ROT_EINVAL;
  if (!(alpha >= 0.0 && alpha <= 1.0)) return ROT_EINVAL;
  if (ideal != ROT_ALPHA_IDEAL_BEFORE && ideal != ROT_ALPHA_IDEAL_AFTER) return ROT_EINVAL;
  uint64_t total = 0;
  for (int32_t i = 0; i < count; ++i) {
    if (work[i] >= kExactLimit - total) return ROT_EINVAL;
    total += work[i];
  }
  try {
    hvec<int64_t> start;
    if (!bucket_starts(bucket_sizes, n_buckets, count, start)) return ROT_EINVAL;
    hvec<uint64_t> bwork((size_t)n_buckets, 0);
    for (int32_t b = 0; b < n_buckets; ++b)
      for (int64_t i = start[(size_t)b]; i < start[(size_t)b] + bucket_sizes[b]; ++i)
        bwork[(size_t)b] += work[i];
    hvec<int32_t> order((size_t)n_buckets);
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      return bwork[(size_t)a] != bwork[(size_t)b] ? bwork[(size_t)a] > bwork[(size_t)b] : a < b;
    });

    const size_t R = (size_t)ranks;
    const double Rd = (double)ranks;
    hvec<uint64_t> L(R, 0);
    hvec<double> deficit(R), share(R);
    hvec<uint64_t> prefix;
    hvec<int64_t> cut(R);
    for (const int32_t b : order) {
      const uint64_t Wb = bwork[(size_t)b];
      const int64_t s0 = start[(size_t)b], nb = bucket_sizes[b];
      uint64_t placed = 0;
      for (size_t r = 0; r < R; ++r) placed += L[r];
      if (ideal == ROT_ALPHA_IDEAL_AFTER) placed += Wb;
      const double target_load = (double)placed / Rd;
      double dsum = 0.0;
      for (size_t r = 0; r < R; ++r) {
        const double d = target_load - (double)L[r];
        deficit[r] = d > 0.0 ? d : 0.0;
        dsum += deficit[r];
      }
      for (size_t r = 0; r < R; ++r) {
        const double fill = dsum > 0.0 ? deficit[r] / dsum : 1.0 / Rd;
        const double even_part = (1.0 - alpha) / Rd;
        const double fill_part = alpha * fill;
        share[r] = even_part + fill_part;
      }
      prefix.assign((size_t)nb + 1, 0);
      for (int64_t j = 0; j < nb; ++j) prefix[(size_t)j + 1] = prefix[(size_t)j] + work[s0 + j];
      // nearest boundary to each cumulative target; the targets increase, so
      // each search may start at the previous cut
      double cum = 0.0;
      int64_t best = 0;
      for (size_t r = 0; r + 1 < R; ++r) {
        cum += share[r];
        const double target = (double)Wb * cum;
        double err = std::fabs((double)prefix[(size_t)best] - target);
        for (int64_t j = best + 1; j <= nb; ++j) {
          const double e = std::fabs((double)prefix[(size_t)j] - target);
          if (e < err) {
            best = j;
            err = e;
          }
        }
        cut[r] = best;
      }
      cut[R - 1] = nb;
      int64_t lo = 0;
      for (size_t r = 0; r < R; ++r) {
        const int64_t hi = std::max(lo, cut[r]);
        for (int64_t j = lo; j < hi; ++j) owners[s0 + j] = (int32_t)r;
        L[r] += prefix[(size_t)hi] - prefix[(size_t)lo];
        lo = hi;
      }
    }
    if (loads)
      for (size_t r = 0; r < R; ++r) loads[r] = L[r];
  } catch (const std::bad_alloc&) {
    return ROT_ENOMEM;
  }
  return ROT_OK;
}

extern "C" int rot_partition_alpha(const uint64_t* work, int32_t count,
                                   const int32_t* bucket_sizes, int32_t n_buckets,
                                   int32_t ranks, double alpha, int32_t* owners,
                                   uint64_t* loads) {
  return rot_partition_alpha_ex(work, count, bucket_sizes, n_buckets, ranks, alpha,
                                ROT_ALPHA_IDEAL_BEFORE, owners, loads);
}
