// Host planner of the pipelined whole-plane forward / input-gradient kernel
// (fwd2_kernel; layout in wtconv_f2.h).  Included by wtconv_api.cu (and by
// the CPU index replay, which checks every plan it makes).
#pragma once

#include <stdint.h>

#include <algorithm>
#include <vector>

#include "wtconv_f2.h"

namespace wt2 {

inline int rup(int a, int b) { return (a + b - 1) / b * b; }
inline int cdiv(int a, int b) { return (a + b - 1) / b; }

inline WtDiv mkdiv(int d) {
  uint32_t s = 0;
  while ((1u << s) < (uint32_t)d) ++s;
  WtDiv f;
  f.shift = s;
  f.mul = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << s) - (uint64_t)d)) / (uint64_t)d + 1);
  return f;
}

// Shared-memory wavefronts of one 16-byte load per item, items taken in
// order by consecutive lanes: per quarter-warp (8 lanes) the largest number
// of distinct 16-byte addresses that share a bank group (address / 16 mod 8).
inline long quarter_wavefronts(const std::vector<int>& offs) {
  long wf = 0;
  for (size_t q = 0; q < offs.size(); q += 8) {
    int cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int seen[8];
    int ns = 0;
    for (size_t i = q; i < offs.size() && i < q + 8; ++i) {
      const int a = offs[i] >> 2;  // 16-byte chunk index
      bool dup = false;
      for (int j = 0; j < ns; ++j) dup |= seen[j] == a;
      if (dup) continue;
      seen[ns++] = a;
      ++cnt[a & 7];
    }
    int m = 0;
    for (int b = 0; b < 8; ++b) m = std::max(m, cnt[b]);
    wf += m;
  }
  return wf;
}

// Strip windows of a (planes x bands x A x T) enumeration in item order.
inline std::vector<int> strip_offsets(int P, int nb, int A, int T, int stride, int band, int plane) {
  std::vector<int> o;
  o.reserve((size_t)P * nb * A * T);
  for (int g = 0; g < P; ++g)
    for (int b = 0; b < nb; ++b)
      for (int r = 0; r < A; ++r)
        for (int s = 0; s < T; ++s) o.push_back(g * plane + b * band + F2_SA * r * stride + 4 * s);
  return o;
}

// Picks (stride, band stride, plane stride) >= the minimum so that the
// enumeration's window loads have the fewest bank conflicts (ties: least
// memory).  rows: allocated rows per band.
inline void pick_strides(int P, int nb, int A, int T, int rows, int min_stride, int& stride, int& band,
                         int& plane, bool tight = false) {
  const int s0 = rup(min_stride, 4);
  if (tight) {  // the smallest layout, whatever its conflicts
    stride = s0;
    band = rows * s0;
    plane = nb * band;
    return;
  }
  long best = -1;
  int bs = s0;
  for (int s = s0; s < s0 + 32; s += 4) {
    const long c = quarter_wavefronts(strip_offsets(P, nb, A, T, s, rows * s, nb * rows * s));
    if (best < 0 || c < best) best = c, bs = s;
  }
  stride = bs;
  const int b0 = rows * stride;
  int bb = b0;
  best = -1;
  if (nb > 1) {
    for (int b = b0; b < b0 + 32; b += 4) {
      const long c = quarter_wavefronts(strip_offsets(P, nb, A, T, stride, b, nb * b));
      if (best < 0 || c < best) best = c, bb = b;
    }
  }
  band = bb;
  const int p0 = nb * band;
  int bp = p0;
  best = -1;
  if (P > 1) {
    for (int p = p0; p < p0 + 32; p += 4) {
      const long c = quarter_wavefronts(strip_offsets(P, nb, A, T, stride, band, p));
      if (best < 0 || c < best) best = c, bp = p;
    }
  }
  plane = bp;
}

// Shared-memory layout of a plan for P planes per unit; returns the bytes.
// tight: 0 = conflict-free strides everywhere; 1 = the smallest Z1 layout;
// 2 = also the smallest B1 layout; 3 = also the smallest X layout.
inline int layout(WtF2Plan& pl, int P, int tight = 0) {
  const int R = pl.K / 2, L = pl.L, NV = f2_nv(pl.K);
  const int es = pl.dtype == 0 ? 4 : 2;
  pl.P = P;
  int off = 0;
  // raw slots
  pl.plane_bytes = pl.H * pl.W * es;
  pl.raw_pb = rup(pl.plane_bytes, 16);
  pl.raw_off = 0;
  pl.raw_slot = rup(P * pl.raw_pb, 128) / 4;
  off = 2 * pl.raw_slot;
  // X: float32 planes, R zero rows above and below, 4 zero columns left and
  // at least R right; rows cover the final strips' windows
  {
    WtF2Buf& X = pl.X;
    X.rows = F2_SA * pl.A[0] + 2 * R;
    const int ms = std::max(4 * (pl.T[0] - 1) + 4 * NV, 4 + pl.W + R);
    pick_strides(P, 1, pl.A[0], pl.T[0], X.rows, ms, X.stride, X.band, X.plane, tight >= 3);
    X.off = off;
    pl.xslot = rup(P * X.plane, 32);
    off += 2 * pl.xslot;
  }
  // bands of every level, margin R
  for (int l = 1; l <= L; ++l) {
    WtF2Buf& B = pl.B[l];
    B.rows = (l == 1 ? F2_SA : F2_SAC) * pl.A[l] + 2 * R;
    const int ms = std::max(4 * (pl.T[l] - 1) + 4 * NV, pl.Ws[l] + 2 * R);
    if (l == 1) {
      pick_strides(P, 4, pl.A[1], pl.T[1], B.rows, ms, B.stride, B.band, B.plane, tight >= 2);
    } else {
      B.stride = rup(ms, 4);
      B.band = B.rows * B.stride;
      B.plane = 4 * B.band;
    }
    B.off = off;
    off += rup(P * B.plane, 32);
  }
  // convolved bands: Z1 (read back by the final strips at level-1 rows up to
  // (F2_SA*A0 - 1) / 2 and columns up to 2*T0 - 1), Zc of levels 2..L
  for (int l = 1; l <= L; ++l) {
    WtF2Buf& Z = pl.Z[l];
    if (l == 1) {
      Z.rows = std::max(F2_SA * pl.A[1], ((F2_SA * pl.A[0] - 1) >> 1) + 1);
      // written at buffer columns zo .. 4*T1 - 1 + zo; read up to level-1
      // column (4*T0 - sh - 1) >> 1, plus zo
      const int ms = std::max(4 * pl.T[1] + pl.zo, ((4 * pl.T[0] - f2_sh(pl.K) - 1) >> 1) + 1 + pl.zo + 1);
      pick_strides(P, 4, pl.A[1], pl.T[1], Z.rows, ms, Z.stride, Z.band, Z.plane, tight >= 1);
    } else {
      Z.rows = F2_SAC * pl.A[l];
      Z.stride = rup(4 * pl.T[l], 4);
      Z.band = Z.rows * Z.stride;
      Z.plane = 4 * Z.band;
    }
    Z.off = off;
    off += rup(P * Z.plane, 32);
  }
  // synthesis cascade sums: levels 2..L-1 (producer only), then R1 (two slots)
  for (int m = 2; m <= L - 1; ++m) {
    WtF2Buf& Rm = pl.RC[m];
    Rm.rows = pl.Hs[m];
    Rm.stride = rup(pl.Ws[m], 4);
    Rm.band = Rm.rows * Rm.stride;
    Rm.plane = Rm.band;
    Rm.off = off;
    off += rup(P * Rm.plane, 32);
  }
  {
    WtF2Buf& R1 = pl.RC[1];
    R1.rows = std::max(pl.Hs[1], ((F2_SA * pl.A[0] - 1) >> 1) + 1);
    R1.stride = rup(std::max(pl.Ws[1] + pl.zo, ((4 * pl.T[0] - f2_sh(pl.K) - 1) >> 1) + 1 + pl.zo + 1), 4);
    R1.band = R1.rows * R1.stride;
    R1.plane = R1.band;
    R1.off = off;
    pl.r1slot = rup(P * R1.plane, 32);
    off += L >= 2 ? 2 * pl.r1slot : 0;
  }
  pl.wb = rup(pl.K * pl.K, 4);
  pl.wslot = rup((1 + 4 * L) * pl.wb, 4);
  pl.w_off = off;
  off += 2 * pl.wslot;
  pl.mb_off = rup(off, 4);
  pl.smem_bytes = 4 * (pl.mb_off + 2 * F2_NMB) + 128;
  return pl.smem_bytes;
}

// Modelled time of a unit of P planes, in cycles of one CTA: the consumer
// group's strip rounds against the producer group's work, whichever is longer.
inline double unit_cost(const WtF2Plan& pl, int P) {
  const double strip = 25.0 * 4 * F2_SA * 1.15;  // a strip's FMAs and overhead, issue slots
  const double back = (cdiv(P * pl.n1, F2_NB) + cdiv(P * pl.nf, F2_NB)) * strip;
  double front = cdiv(P * pl.na, F2_NF) * 90.0 + cdiv(P * pl.nco, F2_NF) * strip * F2_SAC / F2_SA;
  for (int l = 3; l <= pl.L; ++l) front += cdiv(P * pl.Hs[l] * pl.Ws[l], F2_NF) * 40.0 + 60.0;
  for (int l = 2; l <= pl.L; ++l) front += cdiv(P * pl.Hs[l] * pl.Ws[l], F2_NF) * 40.0 + 60.0;
  return std::max(back, front) + 300.0;
}

// Geometry and the planes per unit.  Returns false when the layer does not
// fit two CTAs per SM at one plane per unit (the other kernels take it).
// `smem_per_sm`: bytes of shared memory per SM; ctas_of(plan) -> resident
// CTAs per SM (0: unknown).
template <typename CtasFn>
bool plan(WtF2Plan& pl, int N, int C, int H, int W, int L, int K, int dtype, int smem_per_sm, int max_smem_cta,
          int num_sms, CtasFn ctas_of) {
  pl = WtF2Plan();
  pl.N = N; pl.C = C; pl.H = H; pl.W = W; pl.L = L; pl.K = K; pl.dtype = dtype;
  pl.Hs[0] = H;
  pl.Ws[0] = W;
  for (int l = 1; l <= L; ++l) {
    pl.Hs[l] = (pl.Hs[l - 1] + 1) / 2;
    pl.Ws[l] = (pl.Ws[l - 1] + 1) / 2;
  }
  pl.A[0] = cdiv(H, F2_SA);
  pl.T[0] = cdiv(W + f2_sh(K), 4);
  pl.zo = f2_zo(K);
  for (int l = 1; l <= L; ++l) {
    pl.A[l] = cdiv(pl.Hs[l], l == 1 ? F2_SA : F2_SAC);
    pl.T[l] = cdiv(pl.Ws[l], 4);
  }
  pl.n1 = 4 * pl.A[1] * pl.T[1];
  pl.nf = pl.A[0] * pl.T[0];
  pl.co_begin[2] = 0;
  for (int l = 2; l <= L; ++l) pl.co_begin[l + 1] = pl.co_begin[l] + 4 * pl.A[l] * pl.T[l];
  pl.nco = L >= 2 ? pl.co_begin[L + 1] : 0;
  pl.nbh = cdiv(H, 4);
  pl.nbw = cdiv(W, 4);
  pl.na = pl.nbh * pl.nbw;
  // per-SM budget for two CTAs (1 KB of each CTA's shared memory is reserved)
  const int budget = std::min(smem_per_sm / 2 - 1024 - 64, max_smem_cta);
  // the least tight layout that fits one plane per unit
  int tight = 0;
  while (tight <= 3 && layout(pl, 1, tight) > budget) ++tight;
  if (tight > 3) return false;
  const int pmax = std::max(1, std::min(N, 64));
  int bestP = 1;
  double best = -1;
  for (int P = 1; P <= pmax; ++P) {
    if (layout(pl, P, tight) > budget) break;
    const double c = unit_cost(pl, P) / P;
    if (best < 0 || c < best * 0.98) best = c, bestP = P;
  }
  layout(pl, bestP, tight);
  pl.G = cdiv(N, bestP);
  pl.units = C * pl.G;
  pl.d_n1 = mkdiv(pl.n1);
  pl.d_a1t1 = mkdiv(pl.A[1] * pl.T[1]);
  pl.d_t1 = mkdiv(pl.T[1]);
  pl.d_nf = mkdiv(pl.nf);
  pl.d_tf = mkdiv(pl.T[0]);
  pl.d_na = mkdiv(pl.na);
  pl.d_nbw = mkdiv(pl.nbw);
  pl.d_G = mkdiv(pl.G);
  pl.wait_shift = 31;
  pl.dbg_extra_tx = 0;
  int ctas = ctas_of(pl);
  if (ctas <= 0) ctas = std::max(1, std::min(2, smem_per_sm / (pl.smem_bytes + 1024)));
  const long long slots = (long long)ctas * num_sms;
  pl.grid = (int)std::min<long long>(pl.units, slots);
  return true;
}

// Load mode for the activation pointer: one bulk copy per plane (planes a
// multiple of 16 bytes, pointer 16-byte aligned), else cp.async chunks of 16,
// 8 or 4 bytes.  False if not even 4-byte chunks fit (16-bit planes of an odd
// element count): the other kernels take such layers.
inline bool set_load(WtF2Plan& pl, const void* x) {
  const uintptr_t a = (uintptr_t)x;
  const int pb = pl.plane_bytes;
  if (pb % 16 == 0 && a % 16 == 0) {
    pl.load_mode = 0;
    pl.chunk = 16;
  } else if (pb % 8 == 0 && a % 8 == 0) {
    pl.load_mode = 2;
    pl.chunk = 8;
  } else if (pb % 4 == 0 && a % 4 == 0) {
    pl.load_mode = 3;
    pl.chunk = 4;
  } else {
    return false;
  }
  pl.d_chunks = mkdiv(pb / pl.chunk);
  return true;
}

}  // namespace wt2
