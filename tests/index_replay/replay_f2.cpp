// CPU replay of the memory accesses of the pipelined whole-plane forward /
// input-gradient kernel (fwd2_kernel) for the plans its planner makes (test
// infrastructure; host code only, no GPU).
//
// For each plan the replay walks one unit in each raw/X/R1 slot, phase by
// phase in the kernel's order, forming every index with the same helpers
// the kernel uses (wtconv_f2.h), and checks:
//   - every shared-memory access lies inside its own buffer region, the
//     regions are disjoint and end before the mbarriers;
//   - vector accesses are aligned (16-byte float4, 8-byte float2);
//   - writes touch interiors only (zero margins are never written), and every
//     read of a location some phase writes comes after that write in the
//     same unit (a convolution window reads interiors or never-written
//     margins);
//   - the raw copies and the output stores stay inside x and y;
//   - the persistent CTAs' unit ranges cover every unit once.
//
// Usage:  replay_f2              built-in sweep of layers
//         replay_f2 file CASES   layers "N C H W L k dtype" per line
// Exit status 0 when no check fails.
#include <cstdio>
#include <cstdlib>
#include <string>
#include <vector>

#include "wtconv_f2_plan.h"

static long errors = 0;
static bool g_check_margins = false;  // second sweep: reads of unwritten locations must be margins
#define CHECK(cond, ...)                        \
  do {                                          \
    if (!(cond)) {                              \
      if (errors < 30) {                        \
        printf(__VA_ARGS__);                    \
        printf("\n");                           \
      }                                         \
      ++errors;                                 \
    }                                           \
  } while (0)

struct Region {
  const char* name;
  long lo, hi;  // floats [lo, hi)
};

// Shadow of the dynamic shared memory: which phase last wrote a float (0:
// never), and which region owns it.
struct Shadow {
  std::vector<int> wr;      // phase id of the last write in this unit, 0 = none
  std::vector<char> ever;   // written by any phase of any unit
  std::vector<int> owner;   // region index, -1 = none
  std::vector<Region> regions;
  long size = 0;
  void add(const char* n, long lo, long hi) {
    regions.push_back({n, lo, hi});
  }
  void build(long sz) {
    size = sz;
    owner.assign(sz, -1);
    wr.assign(sz, 0);
    ever.assign(sz, 0);
    for (size_t i = 0; i < regions.size(); ++i) {
      CHECK(regions[i].lo >= 0 && regions[i].hi <= sz && regions[i].lo <= regions[i].hi, "region %s [%ld,%ld) of %ld",
            regions[i].name, regions[i].lo, regions[i].hi, sz);
      for (long a = std::max(0L, regions[i].lo); a < std::min(sz, regions[i].hi); ++a) {
        CHECK(owner[a] < 0, "regions %s and %s overlap at %ld", regions[i].name,
              owner[a] >= 0 ? regions[owner[a]].name : "?", a);
        owner[a] = (int)i;
      }
    }
  }
  int region_of(const char* n) const {
    for (size_t i = 0; i < regions.size(); ++i)
      if (std::string(regions[i].name) == n) return (int)i;
    return -1;
  }
  void w(long a, int n, int phase, int reg, const char* what) {
    CHECK(a >= 0 && a + n <= size, "%s: write [%ld,+%d) outside smem %ld", what, a, n, size);
    if (a < 0 || a + n > size) return;
    if (n == 4) CHECK(a % 4 == 0, "%s: float4 write misaligned at %ld", what, a);
    if (n == 2) CHECK(a % 2 == 0, "%s: float2 write misaligned at %ld", what, a);
    for (int i = 0; i < n; ++i) {
      CHECK(owner[a + i] == reg, "%s: write at %ld in region %d, expected %d", what, a + i, owner[a + i], reg);
      wr[a + i] = phase;
      ever[a + i] = 1;
    }
  }
  // A read that must see data written earlier in this unit, or a margin that
  // no phase ever writes.
  void r(long a, int n, int before_phase, int reg, const char* what) {
    CHECK(a >= 0 && a + n <= size, "%s: read [%ld,+%d) outside smem %ld", what, a, n, size);
    if (a < 0 || a + n > size) return;
    if (n == 4) CHECK(a % 4 == 0, "%s: float4 read misaligned at %ld", what, a);
    if (n == 2) CHECK(a % 2 == 0, "%s: float2 read misaligned at %ld", what, a);
    for (int i = 0; i < n; ++i) {
      CHECK(owner[a + i] == reg, "%s: read at %ld in region %d, expected %d", what, a + i, owner[a + i], reg);
      const int p = wr[a + i];
      CHECK(p != 0 ? p < before_phase : true, "%s: read at %ld of phase %d data before it (phase %d)", what, a + i, p,
            before_phase);
      if (p == 0 && g_check_margins)
        CHECK(!ever[a + i], "%s: read at %ld of a location written only by another unit or a later phase", what,
              a + i);
    }
  }
};

// Second pass: reads of never-written locations are margins only if no phase
// of any unit writes them.
struct ReadLog {
  std::vector<long> addr;
};

static int cases = 0, refused = 0;

static void replay(int N, int C, int H, int W, int L, int K, int dtype) {
  WtF2Plan pl;
  const bool ok = wt2::plan(pl, N, C, H, W, L, K, dtype, 233472, 232448, 152,
                            [](const WtF2Plan& p) { return std::min(2, 233472 / (p.smem_bytes + 1024)); });
  ++cases;
  if (!ok) {
    ++refused;
    return;
  }
  const int R = K / 2, NV = f2_nv(K), KK = K * K, P = pl.P, es = dtype == 0 ? 4 : 2;
  CHECK(pl.smem_bytes <= 232448, "smem %d", pl.smem_bytes);
  CHECK(233472 / (pl.smem_bytes + 1024) >= 2, "fewer than two CTAs per SM");
  CHECK(pl.mb_off % 4 == 0 && 4 * (pl.mb_off + 2 * F2_NMB) + 128 <= pl.smem_bytes, "mbarriers");
  // persistent CTAs cover the units once, in order
  {
    long prev = 0;
    for (int b = 0; b < pl.grid; ++b) {
      const long u0 = (long)pl.units * b / pl.grid, u1 = (long)pl.units * (b + 1) / pl.grid;
      CHECK(u0 == prev && u1 >= u0, "unit ranges");
      prev = u1;
    }
    CHECK(prev == pl.units && pl.grid >= 1 && pl.units == C * pl.G && pl.G * P >= N && (pl.G - 1) * P < N,
          "units %d grid %d", pl.units, pl.grid);
  }
  Shadow sh;
  sh.add("raw0", pl.raw_off, pl.raw_off + pl.raw_slot);
  sh.add("raw1", pl.raw_off + pl.raw_slot, pl.raw_off + 2 * pl.raw_slot);
  sh.add("X0", pl.X.off, pl.X.off + pl.xslot);
  sh.add("X1", pl.X.off + pl.xslot, pl.X.off + 2 * pl.xslot);
  CHECK(P * pl.X.plane <= pl.xslot && pl.X.rows * pl.X.stride <= pl.X.plane, "X slot");
  std::vector<std::string> names;
  names.reserve(64);
  for (int l = 1; l <= L; ++l) {
    names.push_back("B" + std::to_string(l));
    sh.add(names.back().c_str(), pl.B[l].off, pl.B[l].off + (long)P * pl.B[l].plane);
    CHECK(pl.B[l].rows * pl.B[l].stride <= pl.B[l].band && 4 * pl.B[l].band <= pl.B[l].plane, "B%d geometry", l);
  }
  for (int l = 1; l <= L; ++l) {
    names.push_back("Z" + std::to_string(l));
    sh.add(names.back().c_str(), pl.Z[l].off, pl.Z[l].off + (long)P * pl.Z[l].plane);
    CHECK(pl.Z[l].rows * pl.Z[l].stride <= pl.Z[l].band && 4 * pl.Z[l].band <= pl.Z[l].plane, "Z%d geometry", l);
  }
  for (int m = 2; m <= L - 1; ++m) {
    names.push_back("RC" + std::to_string(m));
    sh.add(names.back().c_str(), pl.RC[m].off, pl.RC[m].off + (long)P * pl.RC[m].plane);
  }
  if (L >= 2) {
    sh.add("R1_0", pl.RC[1].off, pl.RC[1].off + pl.r1slot);
    sh.add("R1_1", pl.RC[1].off + pl.r1slot, pl.RC[1].off + 2 * pl.r1slot);
    CHECK(P * pl.RC[1].plane <= pl.r1slot, "R1 slot");
  }
  sh.add("W0", pl.w_off, pl.w_off + pl.wslot);
  sh.add("W1", pl.w_off + pl.wslot, pl.w_off + 2 * pl.wslot);
  CHECK((1 + 4 * L) * pl.wb <= pl.wslot && pl.wb % 4 == 0 && pl.wb >= KK, "weights");
  sh.build(pl.mb_off);
  auto reg = [&](const std::string& n) { return sh.region_of(n.c_str()); };

  const long x_elems = (long)N * C * H * W;
  // Two passes over units in slot 0 and slot 1: a full unit and the last
  // (possibly ragged) unit.  Phase ids increase through a unit.  The whole
  // walk runs twice: the first records every location any phase writes, the
  // second also checks that reads of locations not written in the unit are
  // margins that no phase ever writes.
  for (int sweep = 0; sweep < 2; ++sweep)
  for (int pass = 0; pass < 4; ++pass) {
    g_check_margins = sweep == 1;
    const int slot = pass & 1;
    const int u = pass < 2 ? 0 : pl.units - 1;
    const int c = u / pl.G, n0 = (u - c * pl.G) * P, np = std::min(P, N - n0);
    CHECK(np >= 1, "empty unit");
    std::fill(sh.wr.begin(), sh.wr.end(), 0);
    const int rraw = reg(slot ? "raw1" : "raw0"), rX = reg(slot ? "X1" : "X0"), rW = reg(slot ? "W1" : "W0");
    // copies: raw slot bytes and the source span
    for (int g = 0; g < np; ++g) {
      const long src = ((long)(n0 + g) * C + c) * pl.plane_bytes;
      CHECK(src >= 0 && src + pl.plane_bytes <= x_elems * es, "raw copy source beyond x");
      CHECK((long)g * pl.raw_pb + pl.plane_bytes <= 4L * pl.raw_slot && pl.raw_pb % 16 == 0, "raw copy dest");
      // mark the raw plane written (phase 1); reads check only bounds below
      for (long a = 0; a < (pl.plane_bytes + 3) / 4; ++a)
        sh.w(pl.raw_off + (long)slot * pl.raw_slot + ((long)g * pl.raw_pb) / 4 + a, 1, 1, rraw, "raw copy");
    }
    // weights staged (phase 1)
    for (int i = 0; i < (1 + 4 * L) * pl.wb; ++i) sh.w(pl.w_off + (long)slot * pl.wslot + i, 1, 1, rW, "weights");
    // (1) analysis (phase 2): raw reads, X / B1 / B2 writes
    const int ph_an = 2;
    for (int it = 0; it < np * pl.na; ++it) {
      const int g = wt_fdiv(it, pl.d_na);
      const int rem = it - g * pl.na;
      const int bi = wt_fdiv(rem, pl.d_nbw), bj = rem - bi * pl.nbw;
      CHECK(g == it / pl.na && bi == rem / pl.nbw, "analysis division");
      const int i0 = 4 * bi, j0 = 4 * bj;
      for (int a = 0; a < 4; ++a)
        for (int e = 0; e < 4; ++e) {
          const int i = i0 + a, j = j0 + e;
          if (i < H && j < W) {
            const long byte = (long)g * pl.raw_pb + ((long)i * W + j) * es;
            CHECK(byte + es <= (long)P * pl.raw_pb, "raw read");
            const long fl = pl.raw_off + (long)slot * pl.raw_slot + byte / 4;
            sh.r(fl, 1, ph_an, rraw, "raw read");
          }
        }
      if ((W & 3) == 0 && i0 + 3 < H) {
        const long byte = (long)g * pl.raw_pb + ((long)i0 * W + j0) * es;
        CHECK(byte % (4 * es) == 0, "raw vector read misaligned");
      }
      for (int a = 0; a < 4; ++a) {
        if (i0 + a >= H) continue;
        const long xb = pl.X.off + (long)slot * pl.xslot + (long)g * pl.X.plane + (long)(i0 + a + R) * pl.X.stride + j0 + 4;
        if (j0 + 3 < W) {
          sh.w(xb, 4, ph_an, rX, "X write");
        } else {
          for (int e = 0; e < 4; ++e)
            if (j0 + e < W) sh.w(xb + e, 1, ph_an, rX, "X write");
        }
      }
      for (int pu = 0; pu < 2; ++pu) {
        const int p = 2 * bi + pu, q = 2 * bj;
        if (p >= pl.Hs[1]) continue;
        const long d = f2_at(pl.B[1], g, 0, p, q, R);
        if ((R & 1) == 0 && q + 1 < pl.Ws[1]) {
          for (int b = 0; b < 4; ++b) sh.w(d + (long)b * pl.B[1].band, 2, ph_an, reg("B1"), "B1 write");
        } else {
          for (int qv = 0; qv < 2; ++qv)
            if (q + qv < pl.Ws[1])
              for (int b = 0; b < 4; ++b) sh.w(d + (long)b * pl.B[1].band + qv, 1, ph_an, reg("B1"), "B1 write");
        }
      }
      if (L >= 2) {
        CHECK(bi < pl.Hs[2] && bj < pl.Ws[2], "B2 position");
        const long d = f2_at(pl.B[2], g, 0, bi, bj, R);
        for (int b = 0; b < 4; ++b) sh.w(d + (long)b * pl.B[2].band, 1, ph_an, reg("B2"), "B2 write");
      }
    }
    int ph = 3;
    // (2) levels 3..L
    for (int l = 3; l <= L; ++l, ++ph) {
      const int per = pl.Hs[l] * pl.Ws[l];
      for (int it = 0; it < np * per; ++it) {
        const int g = it / per, rem = it - g * per, p = rem / pl.Ws[l], q = rem - p * pl.Ws[l];
        const long s = f2_at(pl.B[l - 1], g, 0, 2 * p, 2 * q, R);
        const int rs = reg("B" + std::to_string(l - 1));
        sh.r(s, 1, ph, rs, "haar read");
        sh.r(s + 1, 1, ph, rs, "haar read");
        sh.r(s + pl.B[l - 1].stride, 1, ph, rs, "haar read");
        sh.r(s + pl.B[l - 1].stride + 1, 1, ph, rs, "haar read");
        const long d = f2_at(pl.B[l], g, 0, p, q, R);
        for (int b = 0; b < 4; ++b) sh.w(d + (long)b * pl.B[l].band, 1, ph, reg("B" + std::to_string(l)), "haar write");
      }
    }
    // (3) coarse convolutions
    if (L >= 2) {
      for (int it = 0; it < np * pl.nco; ++it) {
        const int g = it / pl.nco;
        int l, b, r, s;
        f2_coarse_strip(pl, it - g * pl.nco, l, b, r, s);
        CHECK(l >= 2 && l <= L && b >= 0 && b < 4 && r >= 0 && r < pl.A[l] && s >= 0 && s < pl.T[l], "coarse strip");
        const long wsrc = pl.w_off + (long)slot * pl.wslot + (1 + 4 * (l - 1) + b) * pl.wb;
        for (int t = 0; t < KK; t += 4) sh.r(wsrc + t, 4, ph, rW, "coarse weights");
        const long win = f2_win(pl.B[l], g, b, r, s, F2_SAC);
        CHECK(win % 4 == 0 && pl.B[l].stride % 4 == 0, "coarse window alignment");
        for (int a = 0; a < F2_SAC + K - 1; ++a)
          for (int v4 = 0; v4 < NV; ++v4)
            sh.r(win + (long)a * pl.B[l].stride + 4 * v4, 4, ph, reg("B" + std::to_string(l)), "coarse window");
        const long zd = pl.Z[l].off + (long)g * pl.Z[l].plane + (long)b * pl.Z[l].band + (long)F2_SAC * r * pl.Z[l].stride + 4 * s;
        for (int o = 0; o < F2_SAC; ++o) sh.w(zd + (long)o * pl.Z[l].stride, 4, ph, reg("Z" + std::to_string(l)), "Zc write");
      }
      ++ph;
      // (4) cascade
      for (int l = L; l >= 2; --l, ++ph) {
        const int per = pl.Hs[l] * pl.Ws[l];
        WtF2Buf Rout = pl.RC[l - 1];
        std::string rout = l == 2 ? (slot ? "R1_1" : "R1_0") : "RC" + std::to_string(l - 1);
        if (l == 2) Rout.off += slot * pl.r1slot + pl.zo;
        for (int it = 0; it < np * per; ++it) {
          const int g = it / per, rem = it - g * per, p = rem / pl.Ws[l], q = rem - p * pl.Ws[l];
          const long z = f2_at(pl.Z[l], g, 0, p, q, 0);
          for (int b = 0; b < 4; ++b) sh.r(z + (long)b * pl.Z[l].band, 1, ph, reg("Z" + std::to_string(l)), "cascade Z");
          if (l < L) {
            const long a = f2_at(pl.RC[l], g, 0, p, q, 0);
            sh.r(a, 1, ph, reg("RC" + std::to_string(l)), "cascade rec");
            CHECK(sh.wr[a] != 0, "cascade reads an unwritten rec");
          }
          const long d = f2_at(Rout, g, 0, 2 * p, 2 * q, 0);
          for (int uu = 0; uu < 2; ++uu)
            for (int vv = 0; vv < 2; ++vv)
              if (2 * p + uu < pl.Hs[l - 1] && 2 * q + vv < pl.Ws[l - 1])
                sh.w(d + (long)uu * Rout.stride + vv, 1, ph, reg(rout), "cascade write");
        }
      }
    }
    // consumers: (a) level-1 convolutions
    const int ph_l1 = ph++;
    for (int k = 0; k < np * pl.n1; ++k) {
      const F2Strip t = f2_l1_strip(pl, k);
      CHECK(t.g == k / pl.n1 && t.b >= 0 && t.b < 4 && t.r >= 0 && t.r < pl.A[1] && t.s >= 0 && t.s < pl.T[1],
            "l1 strip decode");
      const long wsrc = pl.w_off + (long)slot * pl.wslot + (1 + t.b) * pl.wb;
      for (int q4 = 0; q4 < KK; q4 += 4) sh.r(wsrc + q4, 4, ph_l1, rW, "l1 weights");
      const long win = f2_win(pl.B[1], t.g, t.b, t.r, t.s);
      for (int a = 0; a < F2_SA + K - 1; ++a)
        for (int v4 = 0; v4 < NV; ++v4) sh.r(win + (long)a * pl.B[1].stride + 4 * v4, 4, ph_l1, reg("B1"), "l1 window");
      const long zd = pl.Z[1].off + (long)t.g * pl.Z[1].plane + (long)t.b * pl.Z[1].band +
                      (long)F2_SA * t.r * pl.Z[1].stride + 4 * t.s + pl.zo;
      CHECK(4 * t.s + pl.zo + 4 <= pl.Z[1].stride, "Z1 write beyond stride");
      for (int o = 0; o < F2_SA; ++o) {
        const long zr = zd + (long)o * pl.Z[1].stride;
        if (pl.zo == 0) {
          sh.w(zr, 4, ph_l1, reg("Z1"), "Z1 write");
        } else {
          sh.w(zr, 1, ph_l1, reg("Z1"), "Z1 write");
          sh.w(zr + 1, 2, ph_l1, reg("Z1"), "Z1 write");
          sh.w(zr + 3, 1, ph_l1, reg("Z1"), "Z1 write");
        }
      }
    }
    // (b) final strips
    const int ph_f = ph++;
    const int SH = f2_sh(K);
    for (int k = 0; k < np * pl.nf; ++k) {
      const F2Strip t = f2_final_strip(pl, k);
      CHECK(t.g == k / pl.nf && t.r >= 0 && t.r < pl.A[0] && t.s >= 0 && t.s < pl.T[0], "final strip decode");
      const int c0 = 4 * t.s - SH, qb = c0 >> 1;
      for (int o = 0; o < F2_SA; ++o) {
        const int i = F2_SA * t.r + o, p = i >> 1;
        CHECK(p < pl.Z[1].rows && (L < 2 || p < pl.RC[1].rows), "Z1/R1 row beyond rows");
        // the columns this row reads, and which output columns each feeds
        std::vector<std::pair<long, int>> zcols;  // (buffer column, width), level-1 column
        if ((SH & 1) == 0) {
          zcols.push_back({qb + pl.zo, 2});
          CHECK((qb + pl.zo) >= 0 && (qb + pl.zo) % 2 == 0, "synthesis pair column");
        } else {
          for (int d = 0; d < 3; ++d) zcols.push_back({std::max(qb + d, 0) + pl.zo, 1});
        }
        for (auto& zc : zcols) {
          CHECK(zc.first + zc.second <= pl.Z[1].stride && (L < 2 || zc.first + zc.second <= pl.RC[1].stride),
                "synthesis column beyond stride");
          for (int b = 0; b < 4; ++b)
            sh.r(pl.Z[1].off + (long)t.g * pl.Z[1].plane + (long)b * pl.Z[1].band + (long)p * pl.Z[1].stride + zc.first,
                 zc.second, ph_f, reg("Z1"), "Z1 read");
          if (L >= 2)
            sh.r(pl.RC[1].off + (long)slot * pl.r1slot + (long)t.g * pl.RC[1].plane + (long)p * pl.RC[1].stride + zc.first,
                 zc.second, ph_f, reg(slot ? "R1_1" : "R1_0"), "R1 read");
        }
        // every output column inside the plane reads its own level-1 column,
        // which an earlier phase wrote
        for (int j = 0; j < 4; ++j) {
          const int cc = c0 + j;
          if (i >= H || cc < 0 || cc >= W) continue;
          const int q = cc >> 1;
          const int d = (j + (SH & 1)) >> 1;
          CHECK(q == qb + d, "synthesis column mapping");
          for (int b = 0; b < 4; ++b) {
            const long a = pl.Z[1].off + (long)t.g * pl.Z[1].plane + (long)b * pl.Z[1].band + (long)p * pl.Z[1].stride + q + pl.zo;
            CHECK(sh.wr[a] == ph_l1, "valid output reads unwritten Z1");
          }
          if (L >= 2) {
            const long a = pl.RC[1].off + (long)slot * pl.r1slot + (long)t.g * pl.RC[1].plane + (long)p * pl.RC[1].stride + q + pl.zo;
            CHECK(sh.wr[a] != 0, "valid output reads unwritten R1");
          }
        }
      }
      for (int q4 = 0; q4 < KK; q4 += 4) sh.r(pl.w_off + (long)slot * pl.wslot + q4, 4, ph_f, rW, "base weights");
      const long win = pl.X.off + (long)slot * pl.xslot + (long)t.g * pl.X.plane + (long)F2_SA * t.r * pl.X.stride + 4 * t.s;
      for (int a = 0; a < F2_SA + K - 1; ++a)
        for (int v4 = 0; v4 < NV; ++v4) sh.r(win + (long)a * pl.X.stride + 4 * v4, 4, ph_f, rX, "X window");
      for (int o = 0; o < F2_SA; ++o) {
        const int i = F2_SA * t.r + o;
        if (i >= H) continue;
        for (int j = 0; j < 4; ++j) {
          const int jj = c0 + j;
          if (jj < 0 || jj >= W) continue;
          const long e = ((long)(n0 + t.g) * C + c) * H * W + (long)i * W + jj;
          CHECK(e >= 0 && e < x_elems, "y store beyond y");
        }
        const long e0 = ((long)(n0 + t.g) * C + c) * H * W + (long)i * W + c0;
        if ((W & 3) == 0 && SH == 0) CHECK((e0 & 3) == 0, "y 4-element store alignment");
        if ((W & 3) == 0 && SH == 2 && c0 >= 0) CHECK((e0 & 1) == 0, "y 2-element store alignment");
      }
    }
  }
}

int main(int argc, char** argv) {
  std::vector<std::vector<int>> layers;
  if (argc >= 3 && std::string(argv[1]) == "file") {
    FILE* f = fopen(argv[2], "r");
    if (!f) return 2;
    int v[7];
    while (fscanf(f, "%d %d %d %d %d %d %d", &v[0], &v[1], &v[2], &v[3], &v[4], &v[5], &v[6]) == 7)
      layers.push_back(std::vector<int>(v, v + 7));
    fclose(f);
  } else {
    // the benchmark's layers
    const int bench[][7] = {{64, 96, 56, 56, 3, 5, 0},   {2, 32, 32, 32, 2, 5, 0},   {128, 192, 28, 28, 2, 5, 1},
                            {128, 192, 28, 28, 2, 5, 2}, {128, 96, 56, 56, 5, 5, 1}, {128, 192, 28, 28, 4, 5, 1},
                            {128, 384, 14, 14, 3, 5, 1}, {128, 768, 7, 7, 2, 5, 1}};
    for (auto& b : bench) layers.push_back(std::vector<int>(b, b + 7));
    for (int C : {96, 192, 384, 768})
      for (int L = 1; L <= 5; ++L)
        for (int dt = 0; dt <= 1; ++dt) {
          const int H = C == 96 ? 56 : C == 192 ? 28 : C == 384 ? 14 : 7;
          layers.push_back({128, C, H, H, L, 5, dt});
        }
    // small planes at every level count and k, both element sizes (every
    // size up to 40 in one dimension, paired with a spread of the other)
    for (int H = 1; H <= 40; ++H)
      for (int W : {H, (H * 7) % 40 + 1, (H * 13 + 5) % 40 + 1})
        for (int L = 1; L <= 6; ++L)
          for (int K = 3; K <= 9; K += 2)
            for (int dt = 0; dt <= 1; ++dt) layers.push_back({(H + W + L) % 5 + 1, 2, H, W, L, K, dt});
    for (int H : {41, 48, 56, 57, 63, 64, 70, 80, 96})
      for (int L = 1; L <= 8; ++L)
        for (int K = 3; K <= 9; K += 2)
          for (int dt = 0; dt <= 1; ++dt) layers.push_back({3, 2, H, H + (L % 3), L, K, dt});
    // several planes per unit with a ragged last unit
    for (int N : {5, 17, 33, 63})
      for (int H : {7, 14, 28})
        for (int L = 1; L <= 4; ++L) layers.push_back({N, 3, H, H, L, 5, L & 1});
  }
  for (auto& v : layers) replay(v[0], v[1], v[2], v[3], v[4], v[5], v[6]);
  printf("layers: %d, not taken: %d, errors: %ld\n", cases, refused, errors);
  return errors == 0 ? 0 : 1;
}
