// C ABI: state initialisation, the step itself, status and state export.
//
// A step runs micro-group by micro-group (the plan's order), all on the
// caller's stream:
//   momentum     M <- beta1 M + (1 - beta1) G (and G's TF32 split)
//   refresh      M^T; Z = M^T U or M M^T, ...; A_U, A_V; batched QR+ -> U, V
//   rotation     (G V)^T, (M V)^T; G~ = U^T G V, M~ = U^T M V
//   Adam         v <- beta2 v + (1 - beta2) G~^2; D = M~ / (sqrt(v) + eps)
//   back         (D V^T)^T; W <- W - lr U (D V^T)
// Every product is C = A * B^T with both operands K-major, so U, V are kept
// both as-is and transposed, and the intermediates are written in the layout
// their consumer reads.
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "plan.h"
#include "rot_internal.h"

namespace rot {

std::atomic<int> g_nonfinite_check{0};

int gemm_tc(const hvec<GemmProblem>& probs, int precision, int* status,
            cudaStream_t stream);

int gemm_grouped(const hvec<GemmProblem>& probs, int precision, int* status,
                 cudaStream_t stream) {
  return gemm_tc(probs, precision, status, stream);
}

namespace {

inline float* F(void* base, uint64_t off) {
  return reinterpret_cast<float*>(static_cast<char*>(base) + off);
}
inline const float* F(const void* base, uint64_t off) {
  return reinterpret_cast<const float*>(static_cast<const char*>(base) + off);
}

GemmProblem gp(int M, int N, int K, const float* ah, const float* al, int lda, const float* bh,
               const float* bl, int ldb, float* ch, float* cl, int ldc, int epi,
               float alpha = 0.f, int mma_only = 0) {
  GemmProblem P;
  P.mma_only = mma_only;
  P.M = M;
  P.N = N;
  P.K = K;
  P.a_hi = ah;
  P.a_lo = al;
  P.lda = lda;
  P.b_hi = bh;
  P.b_lo = bl;
  P.ldb = ldb;
  P.c_hi = ch;
  P.c_lo = cl;
  P.ldc = ldc;
  P.epi = epi;
  P.alpha = alpha;
  return P;
}

constexpr float kF16Inv = 1.f / 16384.f;  // undoes the bases' fixed 2^14 scale

// A named range on the host timeline for profilers (NVTX: no cost unless a
// tool is attached); closed when the scope ends, early returns included.
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

inline unsigned short* H(void* base, uint64_t off) {
  return reinterpret_cast<unsigned short*>(static_cast<char*>(base) + off);
}
inline const unsigned short* H(const void* base, uint64_t off) {
  return reinterpret_cast<const unsigned short*>(static_cast<const char*>(base) + off);
}

// A 3xF16 problem: a_*, b_* (and c_* for kEpiStoreF16SplitT) are fp16 arrays.
GemmProblem gp16(int M, int N, int K, const unsigned short* ah, const unsigned short* al, int lda,
                 const unsigned short* bh, const unsigned short* bl, int ldb, void* ch, void* cl,
                 int ldc, int epi, float c0, const float* row_inv, const float* in_r,
                 const float* out_r, float alpha = 0.f) {
  GemmProblem P = gp(M, N, K, reinterpret_cast<const float*>(ah), reinterpret_cast<const float*>(al),
                     lda, reinterpret_cast<const float*>(bh), reinterpret_cast<const float*>(bl),
                     ldb, static_cast<float*>(ch), static_cast<float*>(cl), ldc, epi, alpha);
  P.f16 = 1;
  P.c0 = c0;
  P.row_inv = row_inv;
  P.in_r = in_r;
  P.out_r = out_r;
  return P;
}

// A precise 3xF16 problem (kPrecPrecise16): fp16 operands scaled by rows
// (row_inv for A's rows, col_inv for B's) or uniformly (ina, inb), c0 for the
// bases' fixed 2^14; outb scales a fp16 split output.
GemmProblem gpp16(int M, int N, int K, const unsigned short* ah, const unsigned short* al,
                  int lda, const unsigned short* bh, const unsigned short* bl, int ldb, void* ch,
                  void* cl, int ldc, int epi, float c0, const float* row_inv,
                  const float* col_inv, Bound ina, Bound inb, Bound outb) {
  GemmProblem P = gp16(M, N, K, ah, al, lda, bh, bl, ldb, ch, cl, ldc, epi, c0, row_inv, nullptr,
                       nullptr);
  P.col_inv = col_inv;
  P.ina = ina;
  P.inb = inb;
  P.outb = outb;
  return P;
}

}  // namespace

// Is the current device an sm_103 part?  The answer is cached per device
// ordinal (atomics: any host thread may call this); a failing CUDA query
// (no device, no driver) returns ROT_ECUDA and clears CUDA's last error.
int check_device() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cached[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ROT_ECUDA;
  }
  const bool slot = dev >= 0 && dev < kMaxDevices;
  int answer = slot ? cached[dev].load(std::memory_order_acquire) : 0;
  if (answer == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return ROT_ECUDA;
    }
    answer = (major == 10 && minor == 3) ? 1 : -1;
    if (slot) cached[dev].store(answer, std::memory_order_release);
  }
  return answer == 1 ? ROT_OK : ROT_ENOTSUP;
}

// rot_step's host-side argument checks (no device access).
int check_step_args(const rot_plan* plan, float* const* W, const float* const* G,
                    const void* state, const void* work, int32_t refresh, int32_t precision,
                    float rank_rtol) {
  if (!plan) return ROT_EINVAL;
  if (plan->count == 0) return ROT_OK;
  if (!W || !G || !state || !work) return ROT_EINVAL;
  if ((reinterpret_cast<uintptr_t>(state) & 255) || (reinterpret_cast<uintptr_t>(work) & 255))
    return ROT_EINVAL;
  if (precision != ROT_PREC_TF32 && precision != ROT_PREC_3XTF32 &&
      precision != ROT_PREC_3XTF32_PRECISE && precision != ROT_PREC_3XF16)
    return ROT_EINVAL;
  if (!(rank_rtol >= 1e-6f && rank_rtol < 1.f)) return ROT_EINVAL;
  for (int32_t i = 0; i < plan->count; ++i) {
    if (!W[i] || !G[i]) return ROT_EINVAL;
    if (refresh && (plan->shapes[i].m > kQrMaxDim || plan->shapes[i].n > kQrMaxDim))
      return ROT_ENOTSUP;
  }
  return ROT_OK;
}

namespace {

#define ROT_TRY(x)             \
  do {                         \
    const int _e = (x);        \
    if (_e != ROT_OK) return _e; \
  } while (0)

int run_group(const rot_plan* p, size_t g, float* const* W, const float* const* G, void* state,
              void* work, float beta1, float beta2, float eps, float lr, int refresh,
              int precision, float rank_rtol, cudaStream_t s) {
  const hvec<int32_t>& items = p->groups[g];
  const hvec<WorkLayout>& WL = p->work[g];
  int* status = static_cast<int*>(state);
  int* nonfinite = g_nonfinite_check.load(std::memory_order_relaxed) ? status : nullptr;
  const size_t n_items = items.size();

  const bool f16 = precision == ROT_PREC_3XF16;
  const int compact = p->state_format == ROT_STATE_COMPACT;
  const int mt_epi = compact ? kEpiStoreBF16 : kEpiStoreF32;  // M~ as the state keeps it
  Range group_range("rot: micro-group");
  if (kChecked) ROT_TRY(launch_guards(p->guards[g], work, status, false, s));

  // (1) momentum, and the TF32 split of G (3xF16: its scaled fp16 split)
  if (f16) {
    Range range("rot: momentum");
    if (cudaMemsetAsync(F(work, WL[0].g_rmax), 0, 16 * n_items, s) != cudaSuccess)
      return ROT_ECUDA;
    hvec<Momentum16Seg> segs(n_items);
    for (size_t k = 0; k < n_items; ++k) {
      const int i = items[k];
      const ItemLayout& L = p->items[i];
      const WorkLayout& x = WL[k];
      if (!W[i] || !G[i]) return ROT_EINVAL;
      segs[k] = {G[i], F(state, L.mom), H(work, x.g_hi), H(work, x.g_lo),
                 F(work, x.g_rinv), F(work, x.g_rmax), L.m, L.n, L.ldn,
                 refresh ? H(work, x.m16_hi) : nullptr, H(work, x.m16_lo), F(work, x.m_rinv),
                 F(work, x.m_rmax), nullptr, nullptr, compact, F(work, x.m_amax)};
    }
    ROT_TRY(launch_momentum16(segs, beta1, nonfinite, s));
  } else {
    Range range("rot: momentum");
    hvec<MomentumSeg> segs(n_items);
    for (size_t k = 0; k < n_items; ++k) {
      const int i = items[k];
      const ItemLayout& L = p->items[i];
      if (!W[i] || !G[i]) return ROT_EINVAL;
      segs[k] = {G[i], F(state, L.mom), F(work, WL[k].g_hi), F(work, WL[k].g_lo), L.m, L.n,
                 L.ldn, refresh ? F(work, WL[k].m_hi) : nullptr, F(work, WL[k].m_lo), compact};
    }
    ROT_TRY(launch_momentum(segs, beta1, nonfinite, s));
  }

  // (2) basis refresh.  3xF16: the products on the precise kernel's fp16 form.
  // M's operands: its row-scaled split (rows i scaled by s_i, m_rinv) and M^T
  // under one scale below a = *m_amax, the largest |M_ij|.  The intermediates
  // Z and the Gram matrices are stored as fp16 splits under one scale below a
  // bound on their entries, with r = *m_rmax the largest row norm:
  // |(M V)_ij| <= ||M_i|| <= r, |(M^T U)_ij| <= ||M_:j|| <= sqrt(m) a,
  // |(M M^T)_ij| <= r^2, |(M^T M)_ij| <= m a^2 (U, V orthonormal).  A_U^T and
  // A_V^T come out as the QR's TF32 splits, as in the other modes.
  if (refresh) {
    Range range("rot: basis refresh");
    if (f16) {
      hvec<TransposeF16Seg> tr(n_items);
      for (size_t k = 0; k < n_items; ++k) {
        const ItemLayout& L = p->items[items[k]];
        const WorkLayout& x = WL[k];
        tr[k] = {F(state, L.mom), L.ldn, H(work, x.mT_hi), H(work, x.mT_lo), L.ldm, L.m, L.n,
                 F(work, x.m_amax), compact};
      }
      ROT_TRY(launch_transpose16(tr, s));
      hvec<GemmProblem> first, second;
      for (size_t k = 0; k < n_items; ++k) {
        const ItemLayout& L = p->items[items[k]];
        const WorkLayout& x = WL[k];
        const int m = L.m, n = L.n;
        const float* rinv = F(work, x.m_rinv);
        const float* rmax = F(work, x.m_rmax);
        const float* amax = F(work, x.m_amax);
        const unsigned short *Mh = H(work, x.m16_hi), *Ml = H(work, x.m16_lo);  // m x ldn
        const unsigned short *MTh = H(work, x.mT_hi), *MTl = H(work, x.mT_lo);  // n x ldm
        const unsigned short *Uth = H(state, L.ut16_hi), *Utl = H(state, L.ut16_lo);
        const unsigned short *Vth = H(state, L.vt16_hi), *Vtl = H(state, L.vt16_lo);
        unsigned short *Zuh = H(work, x.zu_hi), *Zul = H(work, x.zu_lo);
        unsigned short *Zvh = H(work, x.zv_hi), *Zvl = H(work, x.zv_lo);
        float *Auh = F(work, x.aut_hi), *Aul = F(work, x.aut_lo);
        float *Avh = F(work, x.avt_hi), *Avl = F(work, x.avt_lo);
        const Bound none, bmt{amax, 1.f, 0}, bzv{rmax, 1.f, 0};
        if (n < m) {
          // Z_U = M^T U, stored transposed (m x n);  A_U = M Z_U
          const Bound bz{amax, std::sqrt((float)m), 0};
          first.push_back(gpp16(n, m, m, MTh, MTl, L.ldm, Uth, Utl, L.ldm, Zuh, Zul, x.zu_ld,
                                kEpiStoreF16SplitT, kF16Inv, nullptr, nullptr, bmt, none, bz));
          second.push_back(gpp16(m, m, n, Mh, Ml, L.ldn, Zuh, Zul, x.zu_ld, Auh, Aul, L.ldm,
                                 kEpiStoreSplitT, 1.f, rinv, nullptr, none, bz, none));
        } else {
          // Gram M M^T (m x m, stored transposed);  A_U = Gram U
          const Bound bg{rmax, 1.f, 1};
          first.push_back(gpp16(m, m, n, Mh, Ml, L.ldn, Mh, Ml, L.ldn, Zuh, Zul, x.zu_ld,
                                kEpiStoreF16SplitT, 1.f, rinv, rinv, none, none, bg));
          second.push_back(gpp16(m, m, m, Zuh, Zul, x.zu_ld, Uth, Utl, L.ldm, Auh, Aul, L.ldm,
                                 kEpiStoreSplitT, kF16Inv, nullptr, nullptr, bg, none, none));
        }
        if (m < n) {
          // Z_V = M V, stored transposed (n x m);  A_V = M^T Z_V
          first.push_back(gpp16(m, n, n, Mh, Ml, L.ldn, Vth, Vtl, L.ldn, Zvh, Zvl, x.zv_ld,
                                kEpiStoreF16SplitT, kF16Inv, rinv, nullptr, none, none, bzv));
          second.push_back(gpp16(n, n, m, MTh, MTl, L.ldm, Zvh, Zvl, x.zv_ld, Avh, Avl, L.ldn,
                                 kEpiStoreSplitT, 1.f, nullptr, nullptr, bmt, bzv, none));
        } else {
          // Gram M^T M (n x n, stored transposed);  A_V = Gram V
          const Bound bg{amax, (float)m, 1};
          first.push_back(gpp16(n, n, m, MTh, MTl, L.ldm, MTh, MTl, L.ldm, Zvh, Zvl, x.zv_ld,
                                kEpiStoreF16SplitT, 1.f, nullptr, nullptr, bmt, bmt, bg));
          second.push_back(gpp16(n, n, n, Zvh, Zvl, x.zv_ld, Vth, Vtl, L.ldn, Avh, Avl, L.ldn,
                                 kEpiStoreSplitT, kF16Inv, nullptr, nullptr, bg, none, none));
        }
      }
      ROT_TRY(gemm_grouped(first, kPrecPrecise16, status, s));
      ROT_TRY(gemm_grouped(second, kPrecPrecise16, status, s));
    } else {
      hvec<TransposeSeg> tr(n_items);
      hvec<ToTf32Seg> old_bases;
      for (size_t k = 0; k < n_items; ++k) {
        const ItemLayout& L = p->items[items[k]];
        const WorkLayout& x = WL[k];
        tr[k] = {F(work, x.m_hi), F(work, x.m_lo), L.ldn, F(work, x.mT_hi), F(work, x.mT_lo),
                 L.ldm, L.m, L.n, 1, 1, 1};
        // the products' TF32 operands U^T and V^T (the bases before the refresh)
        old_bases.push_back({H(state, L.ut16_hi), H(state, L.ut16_lo), L.ldm, F(work, x.ut_hi),
                             F(work, x.ut_lo), L.ldm, L.m, L.m});
        old_bases.push_back({H(state, L.vt16_hi), H(state, L.vt16_lo), L.ldn, F(work, x.vt_hi),
                             F(work, x.vt_lo), L.ldn, L.n, L.n});
      }
      ROT_TRY(launch_transpose(tr, s));
      ROT_TRY(launch_to_tf32(old_bases, s));

      hvec<GemmProblem> first, second;
      for (size_t k = 0; k < n_items; ++k) {
        const ItemLayout& L = p->items[items[k]];
        const WorkLayout& x = WL[k];
        const int m = L.m, n = L.n;
        const float *Mh = F(work, x.m_hi), *Ml = F(work, x.m_lo);
        const float *MTh = F(work, x.mT_hi), *MTl = F(work, x.mT_lo);
        float *Zuh = F(work, x.zu_hi), *Zul = F(work, x.zu_lo);
        float *Zvh = F(work, x.zv_hi), *Zvl = F(work, x.zv_lo);
        float *Auh = F(work, x.aut_hi), *Aul = F(work, x.aut_lo);
        float *Avh = F(work, x.avt_hi), *Avl = F(work, x.avt_lo);
        if (n < m) {
          // Z_U = M^T U (n x m), stored transposed (m x n);  A_U = M Z_U
          first.push_back(gp(n, m, m, MTh, MTl, L.ldm, F(work, x.ut_hi), F(work, x.ut_lo), L.ldm,
                             Zuh, Zul, x.zu_ld, kEpiStoreSplitT, 0.f, 1));
          second.push_back(gp(m, m, n, Mh, Ml, L.ldn, Zuh, Zul, x.zu_ld, Auh, Aul, L.ldm,
                              kEpiStoreSplitT));
        } else {
          // Gram M M^T (m x m);  A_U = Gram U
          first.push_back(gp(m, m, n, Mh, Ml, L.ldn, Mh, Ml, L.ldn, Zuh, Zul, x.zu_ld,
                             kEpiStoreSplit, 0.f, 1));
          second.push_back(gp(m, m, m, Zuh, Zul, x.zu_ld, F(work, x.ut_hi), F(work, x.ut_lo),
                              L.ldm, Auh, Aul, L.ldm, kEpiStoreSplitT));
        }
        if (m < n) {
          // Z_V = M V (m x n), stored transposed (n x m);  A_V = M^T Z_V
          first.push_back(gp(m, n, n, Mh, Ml, L.ldn, F(work, x.vt_hi), F(work, x.vt_lo), L.ldn,
                             Zvh, Zvl, x.zv_ld, kEpiStoreSplitT, 0.f, 1));
          second.push_back(gp(n, n, m, MTh, MTl, L.ldm, Zvh, Zvl, x.zv_ld, Avh, Avl, L.ldn,
                              kEpiStoreSplitT));
        } else {
          // Gram M^T M (n x n);  A_V = Gram V
          first.push_back(gp(n, n, m, MTh, MTl, L.ldm, MTh, MTl, L.ldm, Zvh, Zvl, x.zv_ld,
                             kEpiStoreSplit, 0.f, 1));
          second.push_back(gp(n, n, n, Zvh, Zvl, x.zv_ld, F(work, x.vt_hi), F(work, x.vt_lo),
                              L.ldn, Avh, Avl, L.ldn, kEpiStoreSplitT));
        }
      }
      ROT_TRY(gemm_grouped(first, kPrecPrecise, status, s));
      ROT_TRY(gemm_grouped(second, kPrecPrecise, status, s));
    }

    hvec<QrProblem> qp;
    int32_t* ranks = reinterpret_cast<int32_t*>(static_cast<char*>(state) + p->ranks_off);
    for (size_t k = 0; k < n_items; ++k) {
      const int i = items[k];
      const ItemLayout& L = p->items[i];
      const WorkLayout& x = WL[k];
      const int rmax = L.m < L.n ? L.m : L.n;
      for (int side = 0; side < 2; ++side) {
        const int pdim = side == 0 ? L.m : L.n;
        const int ld = side == 0 ? L.ldm : L.ldn;
        char* aux = static_cast<char*>(work) + (side == 0 ? x.aux_u : x.aux_v);
        QrProblem q;
        std::memset(&q, 0, sizeof(q));
        q.at = side == 0 ? Split{F(work, x.aut_hi), F(work, x.aut_lo)}
                         : Split{F(work, x.avt_hi), F(work, x.avt_lo)};
        q.qt = side == 0 ? Split{F(work, x.qut_hi), F(work, x.qut_lo)}
                         : Split{F(work, x.qvt_hi), F(work, x.qvt_lo)};
        qr_bind_aux(q, aux, pdim, rmax);
        q.p = pdim;
        q.ld = ld;
        q.rmax = rmax;
        q.ld_out = ld;
        q.rank_out = ranks + 2 * i + side;
        // the new basis, written by the QR's last pass as the state's fp16
        // copies (hi alone in the compact format, whose lo is the shared zeros)
        q.u16_hi = H(state, side == 0 ? L.u16_hi : L.vb16_hi);
        q.u16_lo = compact ? nullptr : H(state, side == 0 ? L.u16_lo : L.vb16_lo);
        q.ut16_hi = H(state, side == 0 ? L.ut16_hi : L.vt16_hi);
        q.ut16_lo = compact ? nullptr : H(state, side == 0 ? L.ut16_lo : L.vt16_lo);
        qp.push_back(q);
      }
    }
    ROT_TRY(qr_batched(qp, rank_rtol, status, s));
  }

  // (3) rotation: S_G^T = (G V)^T ; G~ = U^T S_G.  M~ = U^T M V is recomputed
  // from M only when the bases change (refresh steps); otherwise it follows
  // M~ <- beta1 M~ + (1 - beta1) G~ inside the Adam kernel, which is the same
  // quantity since U and V are unchanged.  In 3xF16 mode both sides run on
  // the fp16 splits (G's or M's rows scaled by s_r, U and V by 2^14, S_G or
  // S_M by a power of two below its bound, the largest row norm of G or M).
  if (!f16) {
    // the TF32-class modes read TF32 splits of the four basis orientations,
    // made from the state's fp16 copies
    Range range("rot: TF32 bases");
    hvec<ToTf32Seg> cv;
    for (size_t k = 0; k < n_items; ++k) {
      const ItemLayout& L = p->items[items[k]];
      const WorkLayout& x = WL[k];
      cv.push_back({H(state, L.u16_hi), H(state, L.u16_lo), L.ldm, F(work, x.u_hi),
                    F(work, x.u_lo), L.ldm, L.m, L.m});
      cv.push_back({H(state, L.ut16_hi), H(state, L.ut16_lo), L.ldm, F(work, x.ut_hi),
                    F(work, x.ut_lo), L.ldm, L.m, L.m});
      cv.push_back({H(state, L.vb16_hi), H(state, L.vb16_lo), L.ldn, F(work, x.vb_hi),
                    F(work, x.vb_lo), L.ldn, L.n, L.n});
      cv.push_back({H(state, L.vt16_hi), H(state, L.vt16_lo), L.ldn, F(work, x.vt_hi),
                    F(work, x.vt_lo), L.ldn, L.n, L.n});
    }
    ROT_TRY(launch_to_tf32(cv, s));
  }
  {
    Range range("rot: rotation");
    hvec<GemmProblem> a, b;
    for (size_t k = 0; k < n_items; ++k) {
      const ItemLayout& L = p->items[items[k]];
      const WorkLayout& x = WL[k];
      const int m = L.m, n = L.n;
      const float *Vth = F(work, x.vt_hi), *Vtl = F(work, x.vt_lo);
      const float *Uth = F(work, x.ut_hi), *Utl = F(work, x.ut_lo);
      if (f16) {
        a.push_back(gp16(m, n, n, H(work, x.g_hi), H(work, x.g_lo), L.ldn, H(state, L.vt16_hi),
                         H(state, L.vt16_lo), L.ldn, H(work, x.sg_hi), H(work, x.sg_lo), L.ldm,
                         kEpiStoreF16SplitT, kF16Inv, F(work, x.g_rinv), nullptr,
                         F(work, x.g_rmax)));
        b.push_back(gp16(m, n, m, H(state, L.ut16_hi), H(state, L.ut16_lo), L.ldm,
                         H(work, x.sg_hi), H(work, x.sg_lo), L.ldm, F(work, x.gt), nullptr, L.ldn,
                         kEpiStoreF32, kF16Inv, nullptr, F(work, x.g_rmax), nullptr));
      } else {
        a.push_back(gp(m, n, n, F(work, x.g_hi), F(work, x.g_lo), L.ldn, Vth, Vtl, L.ldn,
                       F(work, x.sg_hi), F(work, x.sg_lo), L.ldm, kEpiStoreSplitT, 0.f, 1));
        b.push_back(gp(m, n, m, Uth, Utl, L.ldm, F(work, x.sg_hi), F(work, x.sg_lo), L.ldm,
                       F(work, x.gt), nullptr, L.ldn, kEpiStoreF32));
      }
      if (refresh && f16) {  // the M side as the G side, on M's fp16 split
        a.push_back(gp16(m, n, n, H(work, x.m16_hi), H(work, x.m16_lo), L.ldn,
                         H(state, L.vt16_hi), H(state, L.vt16_lo), L.ldn, H(work, x.sm_hi),
                         H(work, x.sm_lo), L.ldm, kEpiStoreF16SplitT, kF16Inv, F(work, x.m_rinv),
                         nullptr, F(work, x.m_rmax)));
        b.push_back(gp16(m, n, m, H(state, L.ut16_hi), H(state, L.ut16_lo), L.ldm,
                         H(work, x.sm_hi), H(work, x.sm_lo), L.ldm, F(state, L.mt), nullptr,
                         L.ldn, mt_epi, kF16Inv, nullptr, F(work, x.m_rmax), nullptr));
      } else if (refresh) {
        a.push_back(gp(m, n, n, F(work, x.m_hi), F(work, x.m_lo), L.ldn, Vth, Vtl, L.ldn,
                       F(work, x.sm_hi), F(work, x.sm_lo), L.ldm, kEpiStoreSplitT, 0.f, 1));
        b.push_back(gp(m, n, m, Uth, Utl, L.ldm, F(work, x.sm_hi), F(work, x.sm_lo), L.ldm,
                       F(state, L.mt), nullptr, L.ldn, mt_epi));
      }
    }
    ROT_TRY(gemm_grouped(a, precision, status, s));
    ROT_TRY(gemm_grouped(b, precision, status, s));
  }

  // (3') Adam in rotated coordinates; D's split overwrites G's split
  if (f16) {
    Range range("rot: adam");
    hvec<Adam16Seg> segs(n_items);
    for (size_t k = 0; k < n_items; ++k) {
      const ItemLayout& L = p->items[items[k]];
      const WorkLayout& x = WL[k];
      segs[k] = {F(work, x.gt), F(state, L.mt), F(state, L.v), H(work, x.g_hi), H(work, x.g_lo),
                 F(work, x.d_rinv), F(work, x.d_rmax), L.m, L.n, L.ldn, compact};
    }
    ROT_TRY(launch_adam16(segs, beta1, beta2, eps, refresh ? 0 : 1, nonfinite, s));
  } else {
    Range range("rot: adam");
    hvec<AdamSeg> segs(n_items);
    for (size_t k = 0; k < n_items; ++k) {
      const ItemLayout& L = p->items[items[k]];
      const WorkLayout& x = WL[k];
      segs[k] = {F(work, x.gt), F(state, L.mt), F(state, L.v), F(work, x.g_hi), F(work, x.g_lo),
                 L.m, L.n, L.ldn, compact};
    }
    ROT_TRY(launch_adam(segs, beta1, beta2, eps, refresh ? 0 : 1, nonfinite, s));
  }

  // (4) back-rotation: (D V^T)^T into S_G's buffer; W -= lr U (D V^T).  In
  // 3xF16 mode D's rows carry their own scales and (D V^T)^T one below the
  // largest row norm of D.
  {
    Range range("rot: back-rotation and apply");
    hvec<GemmProblem> a, b;
    for (size_t k = 0; k < n_items; ++k) {
      const int i = items[k];
      const ItemLayout& L = p->items[i];
      const WorkLayout& x = WL[k];
      const int m = L.m, n = L.n;
      if (f16) {
        a.push_back(gp16(m, n, n, H(work, x.g_hi), H(work, x.g_lo), L.ldn, H(state, L.vb16_hi),
                         H(state, L.vb16_lo), L.ldn, H(work, x.sg_hi), H(work, x.sg_lo), L.ldm,
                         kEpiStoreF16SplitT, kF16Inv, F(work, x.d_rinv), nullptr,
                         F(work, x.d_rmax)));
        b.push_back(gp16(m, n, m, H(state, L.u16_hi), H(state, L.u16_lo), L.ldm,
                         H(work, x.sg_hi), H(work, x.sg_lo), L.ldm, W[i], nullptr, n, kEpiApply,
                         kF16Inv, nullptr, F(work, x.d_rmax), nullptr, lr));
      } else {
        a.push_back(gp(m, n, n, F(work, x.g_hi), F(work, x.g_lo), L.ldn, F(work, x.vb_hi),
                       F(work, x.vb_lo), L.ldn, F(work, x.sg_hi), F(work, x.sg_lo), L.ldm,
                       kEpiStoreSplitT, 0.f, 1));
        b.push_back(gp(m, n, m, F(work, x.u_hi), F(work, x.u_lo), L.ldm, F(work, x.sg_hi),
                       F(work, x.sg_lo), L.ldm, W[i], nullptr, n, kEpiApply, lr));
      }
    }
    ROT_TRY(gemm_grouped(a, precision, status, s));
    ROT_TRY(gemm_grouped(b, precision, status, s));
  }
  // bounds-checked builds: every guard of the group still holds its pattern
  if (kChecked) ROT_TRY(launch_guards(p->guards[g], work, status, true, s));
  return ROT_OK;
}

}  // namespace
}  // namespace rot

using namespace rot;

extern "C" {

namespace {

int state_init(const rot_plan* plan, void* state, void* stream) {
  if (!plan || !state) return ROT_EINVAL;
  if ((reinterpret_cast<uintptr_t>(state) & 255) != 0) return ROT_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(state, 0, 256, s) != cudaSuccess) return ROT_ECUDA;
  if (cudaMemsetAsync(static_cast<char*>(state) + plan->ranks_off, 0xff,
                      8ull * (uint64_t)(plan->count > 0 ? plan->count : 1), s) != cudaSuccess)
    return ROT_ECUDA;
  const bool compact = plan->state_format == ROT_STATE_COMPACT;
  if (compact && plan->zeros_bytes &&
      cudaMemsetAsync(static_cast<char*>(state) + plan->zeros_off, 0, plan->zeros_bytes, s) !=
          cudaSuccess)
    return ROT_ECUDA;
  hvec<FillSeg> segs;
  for (int32_t i = 0; i < plan->count; ++i) {
    const ItemLayout& L = plan->items[i];
    FillSeg mom{F(state, L.mom), nullptr, L.m, L.n, L.ldn, 0};
    FillSeg mt{F(state, L.mt), nullptr, L.m, L.n, L.ldn, 0};
    mom.f16 = mt.f16 = compact;  // bf16 zero has the fp16 zero's bits
    segs.push_back(mom);
    segs.push_back({F(state, L.v), nullptr, L.m, L.n, L.ldn, 0});
    segs.push_back(mt);
    // U = U^T = I, V = V^T = I as 2^14-scaled fp16 splits
    const uint64_t bases[4][2] = {{L.u16_hi, L.u16_lo}, {L.ut16_hi, L.ut16_lo},
                                  {L.vb16_hi, L.vb16_lo}, {L.vt16_hi, L.vt16_lo}};
    for (int j = 0; j < 4; ++j) {
      const int p = j < 2 ? L.m : L.n, ld = j < 2 ? L.ldm : L.ldn;
      FillSeg f{F(state, bases[j][0]), compact ? nullptr : F(state, bases[j][1]), p, p, ld, 1};
      f.f16 = 1;
      segs.push_back(f);
    }
  }
  return launch_fill(segs, s);
}

}  // namespace

int rot_state_init(const rot_plan* plan, void* state, void* stream) {
  try {
    return state_init(plan, state, stream);
  } catch (const std::bad_alloc&) {
    return ROT_ENOMEM;
  }
}

int rot_step(const rot_plan* plan, float* const* W, const float* const* G, void* state,
             void* work, float beta1, float beta2, float eps, float lr, int32_t refresh,
             int32_t precision, float rank_rtol, void* stream) {
  const int args = check_step_args(plan, W, G, state, work, refresh, precision, rank_rtol);
  if (args != ROT_OK || plan->count == 0) return args;
  const int dev = check_device();
  if (dev != ROT_OK) return dev;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  try {
    for (size_t g = 0; g < plan->groups.size(); ++g) {
      const int e = run_group(plan, g, W, G, state, work, beta1, beta2, eps, lr, refresh != 0,
                              precision, rank_rtol, s);
      if (e != ROT_OK) return e;
    }
  } catch (const std::bad_alloc&) {  // the launch descriptors are host vectors
    return ROT_ENOMEM;
  }
  return ROT_OK;
}

int32_t rot_set_nonfinite_check(int32_t on) {
  return g_nonfinite_check.exchange(on != 0 ? 1 : 0);
}

int rot_status(const rot_plan* plan, void* state, int32_t* status, void* stream) {
  if (!plan || !state || !status) return ROT_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, state, sizeof(host), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ROT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ROT_ECUDA;
  if (host != 0) {
    if (cudaMemsetAsync(state, 0, sizeof(int32_t), s) != cudaSuccess) return ROT_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return ROT_ECUDA;
  }
  *status = host;
  return ROT_OK;
}

int rot_state_export(const rot_plan* plan, const void* state, int32_t item, int32_t which,
                     float* dst, void* stream) {
  if (!plan || !state || !dst || item < 0 || item >= plan->count) return ROT_EINVAL;
  const ItemLayout& L = plan->items[item];
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (which) {
    case ROT_WHICH_M:
      return launch_combine(F(state, L.mom), nullptr, L.ldn, dst, L.n, L.m, L.n, s,
                            plan->state_format == ROT_STATE_COMPACT);
    case ROT_WHICH_V2:
      return launch_combine(F(state, L.v), nullptr, L.ldn, dst, L.n, L.m, L.n, s);
    case ROT_WHICH_U:
      return launch_combine16(H(state, L.u16_hi), H(state, L.u16_lo), L.ldm, dst, L.m, L.m, L.m,
                              s);
    case ROT_WHICH_V:
      return launch_combine16(H(state, L.vb16_hi), H(state, L.vb16_lo), L.ldn, dst, L.n, L.n,
                              L.n, s);
    default:
      return ROT_EINVAL;
  }
}

int rot_state_ranks(const rot_plan* plan, const void* state, int32_t item, int32_t* rank_u,
                    int32_t* rank_v, void* stream) {
  if (!plan || !state || !rank_u || !rank_v || item < 0 || item >= plan->count) return ROT_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t r[2];
  const char* src = static_cast<const char*>(state) + plan->ranks_off + 8ull * item;
  if (cudaMemcpyAsync(r, src, sizeof(r), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ROT_ECUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return ROT_ECUDA;
  *rank_u = r[0];
  *rank_v = r[1];
  return ROT_OK;
}

const char* rot_strerror(int code) {
  switch (code) {
    case ROT_OK: return "ok";
    case ROT_EINVAL: return "invalid argument";
    case ROT_ENOMEM: return "host allocation failed";
    case ROT_ECUDA: return "CUDA error";
    case ROT_ETIMEOUT: return "device-side wait timed out";
    case ROT_ENONFINITE: return "non-finite value";
    case ROT_ENOTSUP: return "device is not sm_103 or feature not built";
    case ROT_ETOOLARGE: return "workspace need exceeds the static no-allocation scratch";
    case ROT_ECORRUPT: return "a workspace guard was overwritten (bounds-checked build)";
    default: return "unknown error";
  }
}

}  // extern "C"
