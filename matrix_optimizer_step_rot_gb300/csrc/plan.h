// Plan object behind the opaque rot_plan handle: groups, owners and the byte
// offsets of every buffer in the caller's state and workspace blobs.
#pragma once

#include <stdint.h>

#include <vector>

#include "rot.h"
#include "rot_internal.h"

namespace rot {

// Offsets (bytes from the state blob's base) of one matrix's state.  Each
// quantity is kept once: M, v and M~ in float32; each basis in the two
// orientations the 3xF16 products read, as scaled fp16 splits
// (hi + lo = 2^14 x, 22 significant bits, the same as the TF32 splits the
// tensor cores read).  TF32 splits are made from them in the workspace where
// a product needs them.
// In the compact format (ROT_STATE_COMPACT) M and M~ are bf16 and each basis
// orientation a single 2^14-scaled fp16 (the lo offsets then all point at
// one shared array of zeros, which the products read as the missing lo).
struct ItemLayout {
  int m, n, ldm, ldn;                 // ldm = pad(m), ldn = pad(n)
  uint64_t mom;                       // momentum M (float32, or bf16), m x ldn
  uint64_t v;                         // second moment (float32), m x ldn
  uint64_t mt;                        // M~ = U^T M V (float32, or bf16), m x ldn
  // fp16 splits of U, U^T (m x ldm) and V, V^T (n x ldn), scaled by 2^14
  uint64_t u16_hi, u16_lo, ut16_hi, ut16_lo;
  uint64_t vb16_hi, vb16_lo, vt16_hi, vt16_lo;
};

// Offsets (bytes from the workspace blob's base) of one matrix's temporaries
// while its micro-group runs.
struct WorkLayout {
  // rotation region
  uint64_t g_hi, g_lo;    // G split (m x ldn); later D split
  uint64_t sg_hi, sg_lo;  // (G V)^T split (n x ldm); later (D V^T)^T split
  uint64_t sm_hi, sm_lo;  // (M V)^T split (n x ldm)
  uint64_t gt, mt;        // G~, M~ float32 (m x ldn)
  // 3xF16: G's and D's fp16 splits live in g_hi / g_lo, (G V)^T's and
  // (D V^T)^T's in sg_hi / sg_lo.  Scale slots: per row of G and of D the
  // inverse of its power-of-two scale (m floats each), and the largest row
  // 2-norm of G and of D (one float each, set by atomic max; the group's
  // row-norm slots are contiguous from WorkLayout of its first item's g_rmax,
  // four floats per item, so one memset clears them).
  uint64_t g_rinv, d_rinv, g_rmax, d_rmax;
  // refresh steps in 3xF16: M's row-scaled fp16 split (m x ldn), its rows'
  // inverse scales, row-norm bound and largest |M_ij| (third and fourth
  // floats of the item's slots)
  uint64_t m16_hi, m16_lo, m_rinv, m_rmax, m_amax;
  // TF32 splits of the bases (made from the fp16 state copies): U^T and
  // V^T for the refresh products; all four for the TF32-class rotation
  // modes.  M's TF32 split on refresh steps.
  uint64_t u_hi, u_lo, ut_hi, ut_lo;  // m x ldm
  uint64_t vb_hi, vb_lo, vt_hi, vt_lo;  // n x ldn
  uint64_t m_hi, m_lo;                // m x ldn
  // refresh region
  uint64_t mT_hi, mT_lo;  // M^T split (n x ldm)
  int zu_rows, zu_ld;
  uint64_t zu_hi, zu_lo;  // (M^T U)^T (m x ldn) or M M^T (m x ldm)
  int zv_rows, zv_ld;
  uint64_t zv_hi, zv_lo;  // (M V)^T (n x ldm) or M^T M (n x ldn)
  uint64_t aut_hi, aut_lo;  // A_U^T split (m x ldm); QR input, then reflectors
  uint64_t avt_hi, avt_lo;  // A_V^T split (n x ldn)
  uint64_t qut_hi, qut_lo;  // Q^T accumulators of the QR, splits
  uint64_t qvt_hi, qvt_lo;
  uint64_t aux_u, aux_v;  // QR scratch
};

uint64_t item_cost(int64_t m, int64_t n);
uint64_t item_bytes(int64_t m, int64_t n);

}  // namespace rot

struct rot_plan {
  int32_t count = 0;
  int32_t ranks = 1;
  int32_t state_format = ROT_STATE_FULL;
  uint64_t zeros_off = 0;    // compact format: the shared zero array (fp16), else 0
  uint64_t zeros_bytes = 0;
  uint64_t c_max = 0;
  rot::hvec<rot_shape> shapes;
  rot::hvec<rot::hvec<int32_t>> groups;
  rot::hvec<uint64_t> group_bytes, group_cost;
  rot::hvec<int32_t> owners;
  // layout
  uint64_t state_bytes = 0, work_bytes = 0;
  uint64_t ranks_off = 0;  // int32 pairs (rank_u, rank_v) per item
  rot::hvec<rot::ItemLayout> items;
  rot::hvec<rot::hvec<rot::WorkLayout>> work;  // [group][position in group]
  // bounds-checked builds (ROT_CHECK): offsets of the 256-byte guard regions
  // after every workspace slice, per micro-group (empty otherwise)
  rot::hvec<rot::hvec<uint64_t>> guards;
};

namespace rot {
void build_groups(rot_plan* p);
void build_layout(rot_plan* p);
}  // namespace rot
