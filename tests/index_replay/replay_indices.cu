// CPU replay of the memory accesses of every kernel, for the launch plans
// the library's own planner produces (test infrastructure; no GPU needed).
//
// The planner (wtconv_api.cu) is compiled in, with the launch functions
// replaced by stubs, so every plan here is exactly what a call would launch.
// For each plan the replay walks the kernels' phases in order and recomputes
// each index they form: input loads and box-copy geometry, the Haar analysis
// reads and writes, the band-convolution and correlation windows, the final
// tiles' reads of the Z buffers and of the input plane (and the 2 x 2 blocks
// of the bands of at most 2 x 2 coefficients), the 16/8-byte vector
// stores to y / dx, the 16-bit staging areas, the mbarrier slots and the CTA
// work ranges and record slots that the gradient finalize searches.  Every
// access must stay inside its buffer, every read of a zero margin must hit a
// location no phase writes, and every read of an interior must hit a
// location an earlier phase wrote.
//
// The replay restates the kernels' index arithmetic; it does not execute the
// kernels.  A kernel change that alters an index must change the replay too.
//
// Usage:  replay_indices              exhaustive small planes, windowed and fused plans
//         replay_indices file CASES   layers "N C H W L k dtype" (dtype 0 f32, 1 f16, 2 bf16)
//
// Exit status 0 when no check fails.
#include "wtconv_api.cu"

#include <cstdio>
#include <string>
#include <vector>

// The launch functions, replaced: planning only.  The register and
// occupancy queries the planner makes answer from tables of each kernel
// instance's registers per thread (ptxas -v of the sources for sm_103a) and
// from shared memory, as the device would, so that the plans replayed here
// are the ones a GB300 runs (a kernel change that alters its registers
// changes these tables too).  Index: (k - 3) / 2, then 0 float32 / 1 16-bit.
namespace wt {
static const int kFwdRegs[4] = {96, 128, 168, 168};
static const int kBwRegs[4][2][3] = {  // bw_kernel <TR 4, MI 1>, <TR 4, MI 2>, <TR 8, MI 1>
    {{76, 80, 76}, {70, 104, 70}},
    {{80, 128, 80}, {80, 128, 80}},
    {{111, 232, 128}, {128, 232, 128}},
    {{200, 232, 208}, {198, 234, 208}}};
static const int kBwWinRegs[4][2][2] = {  // bw_win_kernel TR 4, TR 8
    {{64, 62}, {64, 64}},
    {{128, 80}, {128, 80}},
    {{228, 128}, {228, 128}},
    {{236, 212}, {242, 220}}};
static const int kBwfRegs[4][2] = {{64, 96}, {110, 124}, {194, 128}, {255, 236}};  // bwf_kernel (TR 8)
// CTAs of 256 threads per SM: 228 KB of shared memory (1 KB reserved per
// CTA), 64 K registers allocated per warp in steps of 8 per thread.
static int occ256(int regs, int smem) {
  const int by_smem = 233472 / (smem + 16 + 1024);
  const int by_regs = 65536 / (256 * ((regs + 7) / 8 * 8));
  return by_smem < by_regs ? by_smem : by_regs;
}
static int ki(int k) { return (k - 3) / 2; }
static int di(int dtype) { return dtype == 0 ? 0 : 1; }
cudaError_t launch_fwd(const WtFwdPlan&, const CUtensorMap&, int, bool, const void*, const float*, const float*, const float*,
                       const float*, const float*, void*, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_bwd_weight(const WtBwPlan&, const CUtensorMap&, const CUtensorMap&, int, const void*, const void*, const float*, const float*,
                              const float*, const float*, const float*, float*, float*, float*, float*,
                              float*, float*, cudaStream_t) { return cudaSuccess; }
unsigned int take_fwd_faults() { return 0; }
cudaError_t launch_fwd_win(const WtFwdPlan&, const CUtensorMap&, int, bool, const void*, const float*, const float*, const float*,
                           const float*, const float*, void*, cudaStream_t) { return cudaSuccess; }
unsigned int take_win_faults() { return 0; }
cudaError_t launch_bwd_weight_win(const WtBwPlan&, const CUtensorMap&, const CUtensorMap&, int, const void*, const void*, const float*, const float*,
                                  const float*, const float*, const float*, float*, float*, float*, float*, float*, float*, cudaStream_t) { return cudaSuccess; }
int bw_win_ctas_per_sm(const WtBwPlan& pl, int dtype) {
  return occ256(kBwWinRegs[ki(pl.K)][di(dtype)][pl.tbr == 8 ? 1 : 0], pl.smem_bytes);
}
unsigned int take_bww_faults() { return 0; }
int bw_win_regs(int k, int tbr, int dtype) { return kBwWinRegs[ki(k)][di(dtype)][tbr == 8 ? 1 : 0]; }
int fwd_regs(int k, int) { return kFwdRegs[ki(k)]; }
cudaError_t launch_bwd_fused(const WtBwPlan&, const WtFwdPlan&, const CUtensorMap&, const CUtensorMap&, int, const void*, const void*, const float*, const float*,
                             const float*, const float*, const float*, void*, float*, float*, float*, float*, float*, float*, cudaStream_t) { return cudaSuccess; }
int bwf_ctas_per_sm(const WtBwPlan& pl, const WtFwdPlan& fp, int dtype) {
  if (fp.ftp != WT_TP / 2 || pl.tbr != 8) return 0;  // no instance for other tiles
  return occ256(kBwfRegs[ki(pl.K)][di(dtype)], pl.smem_bytes);
}
unsigned int take_bwf_faults() { return 0; }
int bw_regs(int k, int mi, int dtype) { return kBwRegs[ki(k)][di(dtype)][mi == 1 ? 0 : 1]; }  // (the TR 4 instances)
int bw_ctas_per_sm(const WtBwPlan& pl, int dtype) {
  return occ256(kBwRegs[ki(pl.K)][di(dtype)][pl.tbr == 8 ? 2 : pl.mi == 1 ? 0 : 1], pl.smem_bytes);
}
unsigned int take_bw_faults() { return 0; }
cudaError_t launch_lowpass(int, const void*, float*, long long, int, int, int, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_add_carry(int, void*, const float*, long long, int, int, int, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_scale(const float*, float*, int, float, cudaStream_t) { return cudaSuccess; }
}

static long errors = 0;  // failed checks (the first 20 are printed)
static int g_dtype = 0;   // element type of the whole-plane plans: 0 float32, 1 16-bit
#define CHECK(cond, ...) do { if (!(cond)) { if (errors < 20) { printf(__VA_ARGS__); printf("\n"); } ++errors; } } while (0)

// An access to element (pr, pc) of band bi of buffer b, inside a region of plane_floats floats.
static void acc_buf(const WtBuf& b, int nb, int bi, int pr, int pc, int plane_floats, const char* what) {
  const int rows = b.band / b.stride;
  CHECK(bi >= 0 && bi < nb, "%s band %d", what, bi);
  CHECK(pr >= 0 && pr < rows, "%s row %d rows %d", what, pr, rows);
  CHECK(pc >= 0 && pc < b.stride, "%s col %d stride %d", what, pc, b.stride);
  long idx = (long)b.off + (long)bi * b.band + (long)pr * b.stride + pc;
  CHECK(idx >= 0 && idx < plane_floats, "%s idx %ld plane %d", what, idx, plane_floats);
}


// The fused level-1/2 pass over 16-bit raw planes (rows of even length):
// each block of the level-2 grid reads its rows of the raw plane (its first
// column inside the plane) in 4-element groups (8-byte loads, 16-byte
// stores) when rows are whole groups, else in pairs (4-byte loads, 8-byte
// stores; a pair past the row is skipped), and writes the float32 interior
// of buffer X; together the blocks write every interior element once.
static void check_widen12(int H, int W, int H2, int W2, const WtBuf X, int lim) {
  std::vector<int> cnt(lim, 0);
  const int vec = W % 4 == 0 ? 4 : 2;
  CHECK(W % 2 == 0 && X.pcol % vec == 0 && X.stride % vec == 0 && X.off % vec == 0 && (H * W) % vec == 0, "widen12 alignment");
  for (int P = 0; P < H2; ++P) for (int Q = 0; Q < W2; ++Q) {
    CHECK(4 * Q < W, "block's first column inside the plane");
    for (int a = 0; a < 4; ++a) {
      const int i = 4 * P + a;
      if (i >= H) continue;
      for (int e0 = 0; e0 < 4; e0 += vec) {
        if (4 * Q + e0 >= W) { CHECK(vec == 2, "widen12 vector beyond the row"); continue; }
        CHECK((i * W + 4 * Q + e0) % vec == 0 && (X.off + (i + X.prow) * X.stride + 4 * Q + e0 + X.pcol) % vec == 0,
              "widen12 vector alignment");
        for (int e = e0; e < e0 + vec; ++e) {
          const int j = 4 * Q + e;
          CHECK(j < W, "widen12 element beyond the row");
          CHECK(i * W + j < H * W, "widen12 staging read");
          acc_buf(X, 1, 0, i + X.prow, j + X.pcol, lim, "widen12 write");
          const long k = X.off + (long)(i + X.prow) * X.stride + j + X.pcol;
          if (k >= 0 && k < lim) cnt[k]++;
        }
      }
    }
  }
  for (int i = 0; i < H; ++i) for (int j = 0; j < W; ++j)
    CHECK(cnt[X.off + (i + X.prow) * X.stride + j + X.pcol] == 1, "widen12 writes each interior element once");
}

static void check_fwd(int N, int C, int H, int W, int L, int K) {
  wtconv_desc_t d{N, C, H, W, L, K, (wtconv_dtype_t)g_dtype};
  WtFwdPlan pl;
  if (plan_fwd(&d, pl) != WTCONV_OK) return;  // beyond one CTA: the windowed plan takes the layer
  const int R = K / 2, TP = pl.ftp, TQ = WT_TQ, ZT = WT_ZT, PF = pl.wf, XF = pl.xf;
  CHECK(TP == WT_TP || TP == WT_TP / 2, "final tile height");
  CHECK(pl.w_off + (1 + 4 * L) * pl.w_band <= pl.smem_bytes / 4, "weights beyond smem");
  CHECK(pl.P * XF <= pl.xslot && pl.xslot % 32 == 0 && pl.stage_off == pl.xslot &&
        (pl.nsets == 2 ? pl.work_off == 2 * pl.xslot : pl.work_off >= pl.xslot) && pl.work_off % 32 == 0, "input sets");
  CHECK(pl.work_off + pl.P * PF <= pl.w_off, "regions overlap");
  CHECK(pl.mb_off % 2 == 0 && pl.mb_off >= pl.w_off + (1 + 4 * L) * pl.w_band && 4 * pl.mb_off + 16 <= pl.smem_bytes, "mbarriers");
  // TMA box: (stride, rows, 1, P) floats starting at (-4, -R) covers each plane buffer exactly
  CHECK(pl.lev[0].off == 0 && XF == pl.lev[0].band && pl.lev[0].pcol == 4 && pl.lev[0].prow == R, "box = plane buffer");
  CHECK(pl.tma_bytes == 4u * pl.P * XF, "tma bytes");
  if ((W % 4) == 0 && pl.lev[0].stride <= 256 && pl.lev[0].band / pl.lev[0].stride <= 256)
    CHECK(pl.lev[0].stride % 4 == 0, "box inner extent");
  CHECK(pl.smem_bytes <= 232448, "smem too large");
  CHECK(pl.w_off % 4 == 0 && pl.w_band % 4 == 0 && PF % 4 == 0 && XF % 4 == 0 && pl.work_off % 4 == 0, "alignment");
  CHECK(pl.lev[0].pcol % 4 == 0 && pl.lev[0].off % 4 == 0 && pl.lev[0].stride % 4 == 0, "X align");
  if (g_dtype != 0) {  // 16-bit bulk staging in the second input set
    set_bulk(pl, &d, (const void*)(uintptr_t)4096, 4L * (pl.work_off - pl.stage_off));
    if (pl.use_bulk) {
      CHECK((long)pl.P * H * W * 2 <= 4L * (pl.work_off - pl.stage_off), "staging beyond its region");
      CHECK(pl.bulk_bytes % (pl.use_bulk == 1 ? 16 : 8) == 0 && (pl.xslot * 4) % 128 == 0, "staging alignment");
      if (pl.wd_vec == 4) CHECK(W % 4 == 0 && (H * W) % 4 == 0, "widen vector alignment");
      if (pl.wd_vec == 2) CHECK(W % 2 == 0 && pl.lev[0].pcol % 2 == 0 && pl.lev[0].stride % 2 == 0 && XF % 2 == 0, "widen pair alignment");
      CHECK(pl.wd_vec == (W % 4 == 0 ? 4 : W % 2 == 0 ? 2 : 1), "widen item width");
      for (int g = 0; g < pl.P; ++g) CHECK(((long)g * H * W * 2) % (pl.use_bulk == 1 ? 16 : 8) == 0, "staging plane alignment");
      if (L >= 2 && W % 2 == 0) check_widen12(H, W, pl.Hs[2], pl.Ws[2], pl.lev[0], XF);
    }
  }
  std::vector<char> written(PF, 0), xwritten(XF, 0);  // interior writes, to check margins stay zero
  auto wr = [&](const WtBuf& b, int nb, int bi, int pr, int pc, const char* what) {
    acc_buf(b, nb, bi, pr, pc, PF, what);
    long idx = (long)b.off + (long)bi * b.band + (long)pr * b.stride + pc;
    if (idx >= 0 && idx < PF) written[idx] = 1;
  };
  for (int i = 0; i < H; ++i) for (int j = 0; j < W; ++j) { acc_buf(pl.lev[0], 1, 0, i + R, j + 4, XF, "load"); xwritten[pl.lev[0].off + (i + R) * pl.lev[0].stride + j + 4] = 1; }
  // analysis
  if (L == 1) {
    for (int p = 0; p < pl.Hs[1]; ++p) for (int q = 0; q < pl.Ws[1]; ++q) {
      for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) {
        acc_buf(pl.lev[0], 1, 0, 2 * p + u + R, 2 * q + v + 4, XF, "ana1-read");
        if (!(2 * p + u < H && 2 * q + v < W)) CHECK(!xwritten[pl.lev[0].off + (2 * p + u + R) * pl.lev[0].stride + 2 * q + v + 4], "ana1 reads non-zero margin");
      }
      for (int b = 0; b < 4; ++b) wr(pl.lev[1], 4, b, p + pl.lev[1].prow, q + pl.lev[1].pcol, "ana1-write");
    }
  } else {
    for (int P = 0; P < pl.Hs[2]; ++P) for (int Q = 0; Q < pl.Ws[2]; ++Q) {
      for (int a = 0; a < 4; ++a) for (int e = 0; e < 4; ++e) {
        acc_buf(pl.lev[0], 1, 0, 4 * P + a + R, 4 * Q + e + 4, XF, "ana12-read");
        if (!(4 * P + a < H && 4 * Q + e < W)) CHECK(!xwritten[pl.lev[0].off + (4 * P + a + R) * pl.lev[0].stride + 4 * Q + e + 4], "ana12 reads non-zero margin");
      }
      for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) {
        const int p = 2 * P + u, q = 2 * Q + v;
        if (p < pl.Hs[1] && q < pl.Ws[1]) for (int b = 0; b < 4; ++b) wr(pl.lev[1], 4, b, p + pl.lev[1].prow, q + pl.lev[1].pcol, "ana12-w1");
      }
      for (int b = 0; b < 4; ++b) wr(pl.lev[2], 4, b, P + pl.lev[2].prow, Q + pl.lev[2].pcol, "ana12-w2");
    }
  }
  for (int l = 3; l <= L; ++l) {
    const WtBuf S = pl.lev[l - 1], D = pl.lev[l];
    for (int p = 0; p < pl.Hs[l]; ++p) for (int q = 0; q < pl.Ws[l]; ++q) {
      for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) {
        acc_buf(S, 4, 0, 2 * p + u + S.prow, 2 * q + v + S.pcol, PF, "ana-read");
        if (!(2 * p + u < pl.Hs[l - 1] && 2 * q + v < pl.Ws[l - 1])) CHECK(!written[S.off + (2 * p + u + S.prow) * S.stride + 2 * q + v + S.pcol], "ana reads non-zero margin");
      }
      for (int b = 0; b < 4; ++b) wr(D, 4, b, p + D.prow, q + D.pcol, "ana-write");
    }
  }
  // band convolutions: windows must only see interior or untouched zero margin (true by construction: writes only interiors)
  for (int l = 1; l <= L; ++l) {
    const int NV = (ZT + K - 1 + 3) / 4;
    if (pl.Hs[l] <= 2 && pl.Ws[l] <= 2) {  // tiny band: the 2x2 block at its interior origin, then its Z values
      const WtBuf Y = pl.lev[l];
      for (int b = 0; b < 4; ++b) {
        for (int i = 0; i < 2; ++i) for (int j = 0; j < 2; ++j) {
          acc_buf(Y, 4, b, i + Y.prow, j + Y.pcol, PF, "tiny-read");
          if (!(i < pl.Hs[l] && j < pl.Ws[l])) CHECK(!written[Y.off + (long)b * Y.band + (i + Y.prow) * Y.stride + j + Y.pcol], "tiny reads non-zero margin");
        }
        for (int i = 0; i < pl.Hs[l]; ++i) for (int j = 0; j < pl.Ws[l]; ++j) wr(pl.zb[l], 4, b, i, j, "zconv-write");
      }
      continue;
    }
    for (int b = 0; b < 4; ++b) for (int tp = 0; tp < pl.ztr[l]; ++tp) for (int tq = 0; tq < pl.ztc[l]; ++tq) {
      const int p0 = tp * ZT, q0 = tq * ZT;
      for (int a = 0; a < ZT + K - 1; ++a) for (int c = 0; c < 4 * NV; ++c) acc_buf(pl.lev[l], 4, b, p0 + a, q0 + c, PF, "zconv-read");
      for (int o = 0; o < ZT; ++o) for (int j = 0; j < ZT; ++j)
        if (p0 + o < pl.Hs[l] && q0 + j < pl.Ws[l]) wr(pl.zb[l], 4, b, p0 + o, q0 + j, "zconv-write");
    }
    CHECK(pl.zb[l].off % 4 == 0 && pl.zb[l].stride % 4 == 0 && pl.zb[l].band % 4 == 0, "zb align");
  }
  // final tiles
  for (int tp = 0; tp < pl.ftr; ++tp) for (int tq = 0; tq < pl.ftc; ++tq) {
    const int p0 = tp * TP, q0 = tq * TQ;
    if (L >= 2) for (int b = 0; b < 4; ++b) for (int k = 0; k < TP / 2; ++k) acc_buf(pl.zb[2], 4, b, (p0 >> 1) + k, q0 >> 1, PF, "f-z2");
    for (int l = 3; l <= L; ++l) for (int b = 0; b < 4; ++b) acc_buf(pl.zb[l], 4, b, p0 >> (l - 1), q0 >> (l - 1), PF, "f-zl");
    for (int o = 0; o < TP; ++o) for (int b = 0; b < 4; ++b) for (int j = 0; j < TQ; ++j) acc_buf(pl.zb[1], 4, b, p0 + o, q0 + j, PF, "f-z1");
    const int OFF = 4 - R;
    for (int a = 0; a < 2 * TP + K - 1; ++a) for (int c = 0; c < 2 * TQ + K - 1; ++c) acc_buf(pl.lev[0], 1, 0, 2 * p0 + a, 2 * q0 + OFF + c, XF, "f-base");
    // global stores: vector path covers [j0, j0 + 2TQ) with one access of 2TQ*esize bytes
    for (int es = 2; es <= 4; es += 2) {
      const bool vec = (W % (16 / es)) == 0;  // vec_ok with aligned base
      const int j0 = 2 * q0;
      const int bytes = 2 * TQ * es;
      for (int oo = 0; oo < 2 * TP; ++oo) {
        const int i = 2 * p0 + oo;
        if (i >= H) continue;
        if (vec && j0 + 2 * TQ <= W) {
          const long start = ((long)i * W + j0) * es;  // byte offset in the plane (plane base is 16B aligned)
          CHECK(bytes == 16 || bytes == 8 || bytes < 8, "store width");
          if (bytes == 16 || bytes == 8) CHECK(start % bytes == 0, "misaligned vector store es=%d W=%d j0=%d", es, W, j0);
          CHECK(j0 + 2 * TQ <= W, "vector store beyond row");
        }
      }
    }
    // valid outputs must read only valid Z positions
    for (int o = 0; o < TP; ++o) for (int j = 0; j < TQ; ++j) {
      const int p = p0 + o, q = q0 + j;
      if (2 * p >= H || 2 * q >= W) continue;
      CHECK(p < pl.Hs[1] && q < pl.Ws[1], "valid output maps outside level 1");
    }
  }
  CHECK((long)pl.groups * pl.P >= N, "groups do not cover N");
}

static void check_bw(int N, int C, int H, int W, int L, int K) {
  wtconv_desc_t d{N, C, H, W, L, K, (wtconv_dtype_t)g_dtype};
  WtBwPlan pl;
  if (plan_bw(&d, pl) != WTCONV_OK) return;  // beyond one CTA: the windowed plan takes the layer
  const int R = K / 2, BT = WT_BT, WF = pl.wf, KK = K * K;
  const int XB = pl.xbf, DB = pl.dbf;
  CHECK(pl.P * XB <= pl.xr && pl.xr % 32 == 0 && pl.xr + pl.P * DB <= pl.islot && pl.islot % 32 == 0, "input set");
  CHECK((pl.nsets == 1 || pl.nsets == 2) &&
        (pl.stage_off ? (pl.stage_off == pl.nsets * pl.islot && pl.stage_off + pl.P * H * W <= pl.work_off &&
                         pl.stage_off % 32 == 0)
                      : pl.work_off == pl.nsets * pl.islot), "work_off / staging");
  if (g_dtype != 0 && pl.stage_off) {
    set_bulk(pl, &d, (const void*)(uintptr_t)4096, 4L * (pl.work_off - pl.stage_off) / 2);
    CHECK(pl.use_bulk && pl.bulk_bytes % 8 == 0 && (pl.use_bulk == 2 || 2L * pl.P * pl.bulk_bytes < (1L << 20)), "bw staging eligibility");
    CHECK(2L * pl.P * H * W * 2 <= 4L * (pl.work_off - pl.stage_off), "bw staging capacity");
    if (pl.wd_vec == 4) CHECK(pl.ds[0].pcol % 4 == 0 && pl.xs[0].pcol % 4 == 0 && W % 4 == 0, "bw widen alignment");
    if (pl.wd_vec == 2) CHECK(pl.ds[0].pcol % 2 == 0 && pl.xs[0].pcol % 2 == 0 && pl.xs[0].stride % 2 == 0 && pl.ds[0].stride % 2 == 0 && W % 2 == 0 && XB % 2 == 0 && DB % 2 == 0, "bw widen pair alignment");
    CHECK(pl.nsets == 1, "16-bit uses one input set");
    if (L >= 2 && W % 4 == 0) {
      check_widen12(H, W, pl.Hs[2], pl.Ws[2], pl.xs[0], XB);
      check_widen12(H, W, pl.Hs[2], pl.Ws[2], pl.ds[0], DB);
    }
  }
  CHECK(pl.P * WF <= pl.red_floats && pl.red_floats % 4 == 0 && pl.work_off + pl.red_floats == pl.mb_off, "work region");
  CHECK(pl.P * pl.items_per_plane * (KK + 1) <= pl.red_floats, "reduction beyond work region");
  CHECK(pl.mb_off % 2 == 0 && 4 * pl.mb_off + 16 <= pl.smem_bytes && pl.smem_bytes <= 232448, "mbarriers/smem");
  CHECK(pl.mi == 1 || (pl.tbr == 4 && pl.mi == WT_BW_MAX_ITEMS), "tiles per thread");
  CHECK(pl.P * pl.items_per_plane <= pl.mi * WT_BW_THREADS, "items beyond slots");
  CHECK(XB % 4 == 0 && DB % 4 == 0 && WF % 4 == 0 && pl.xs[0].off == 0 && pl.ds[0].off == 0, "align");
  CHECK(pl.xs[0].pcol == 4 && pl.xs[0].prow == R && pl.ds[0].pcol == 0 && pl.ds[0].prow == 0, "level-0 margins");
  CHECK(XB == pl.xs[0].band && DB == pl.ds[0].band, "box = plane buffer");
  CHECK(pl.tma_bytes == 4u * pl.P * (XB + DB), "tma bytes");
  CHECK(pl.xs[0].stride % 4 == 0 && pl.ds[0].stride % 4 == 0, "box inner extent");
  std::vector<char> xw(XB, 0), dw(DB, 0);
  for (int i = 0; i < H; ++i) for (int j = 0; j < W; ++j) {
    acc_buf(pl.xs[0], 1, 0, i + R, j + 4, XB, "load-x");
    acc_buf(pl.ds[0], 1, 0, i, j, DB, "load-dy");
    xw[(i + R) * pl.xs[0].stride + j + 4] = 1;
    dw[i * pl.ds[0].stride + j] = 1;
  }
  for (int s = 0; s < 2; ++s) {
    const WtBuf S0 = s ? pl.ds[0] : pl.xs[0];
    const int IS = s ? DB : XB;
    std::vector<char>& xw_ = s ? dw : xw;
    const WtBuf* D = s ? pl.ds : pl.xs;
    if (L == 1) {
      for (int p = 0; p < pl.Hs[1]; ++p) for (int q = 0; q < pl.Ws[1]; ++q) {
        for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) {
          acc_buf(S0, 1, 0, 2 * p + u + S0.prow, 2 * q + v + S0.pcol, IS, "ana1-read");
          if (!(2 * p + u < H && 2 * q + v < W)) CHECK(!xw_[S0.off + (2 * p + u + S0.prow) * S0.stride + 2 * q + v + S0.pcol], "ana1 margin");
        }
        for (int b = 0; b < 4; ++b) acc_buf(D[1], 4, b, p + D[1].prow, q + D[1].pcol, WF, "ana1-write");
      }
    } else {
      for (int P = 0; P < pl.Hs[2]; ++P) for (int Q = 0; Q < pl.Ws[2]; ++Q) {
        for (int a = 0; a < 4; ++a) for (int e = 0; e < 4; ++e) {
          acc_buf(S0, 1, 0, 4 * P + a + S0.prow, 4 * Q + e + S0.pcol, IS, "ana12-read");
          if (!(4 * P + a < H && 4 * Q + e < W)) CHECK(!xw_[S0.off + (4 * P + a + S0.prow) * S0.stride + 4 * Q + e + S0.pcol], "ana12 margin");
        }
        for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) {
          const int p = 2 * P + u, q = 2 * Q + v;
          if (p < pl.Hs[1] && q < pl.Ws[1]) for (int b = 0; b < 4; ++b) acc_buf(D[1], 4, b, p + D[1].prow, q + D[1].pcol, WF, "ana12-w1");
        }
        for (int b = 0; b < 4; ++b) acc_buf(D[2], 4, b, P + D[2].prow, Q + D[2].pcol, WF, "ana12-w2");
      }
    }
    for (int l = 3; l <= L; ++l)
      for (int p = 0; p < pl.Hs[l]; ++p) for (int q = 0; q < pl.Ws[l]; ++q) {
        for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v)
          acc_buf(D[l - 1], 4, 0, 2 * p + u + D[l - 1].prow, 2 * q + v + D[l - 1].pcol, WF, "ana-read");
        for (int b = 0; b < 4; ++b) acc_buf(D[l], 4, b, p + D[l].prow, q + D[l].pcol, WF, "ana-write");
      }
  }
  for (int item = 0; item < pl.items_per_plane; ++item) {
    int l = 0;
    while (l < L && item >= pl.item_begin[l + 1]) ++l;
    const int tiles = pl.tr[l] * pl.tc[l];
    const int rel = item - pl.item_begin[l];
    const int b = rel / tiles, t = rel - b * tiles;
    const int tp = t / pl.tc[l];
    const int TCW = pl.tcw, TBR = pl.tbr;
    const int p0 = tp * TBR, q0 = (t - tp * pl.tc[l]) * TCW;
    const int nb = l == 0 ? 1 : 4;
    CHECK(b < nb, "item band %d >= %d", b, nb);
    if (l == 0) {  // window columns q0 + (4-R) + c, c < TC+K-1; interior column = that - 4
      for (int a = 0; a < TBR + K - 1; ++a) for (int c = 0; c < TCW + K - 1; ++c) {
        acc_buf(pl.xs[0], 1, 0, p0 + a, q0 + 4 - R + c, XB, "corr-x0");
        const int ii = p0 + a - R, jj = q0 + c - R;
        const long idx = (long)(p0 + a) * pl.xs[0].stride + q0 + 4 - R + c;
        if (!(ii >= 0 && ii < H && jj >= 0 && jj < W) && idx >= 0 && idx < XB) CHECK(!xw[idx], "corr-x0 reads data outside interior");
        if (ii >= 0 && ii < H && jj >= 0 && jj < W && idx >= 0 && idx < XB) CHECK(xw[idx], "corr-x0 maps interior wrong");
      }
      for (int o = 0; o < TBR; ++o) for (int c = 0; c < TCW; ++c) acc_buf(pl.ds[0], 1, 0, p0 + o, q0 + c, DB, "corr-d0");
    } else if (pl.Hs[l] <= 2 && pl.Ws[l] <= 2) {  // tiny band: 2x2 blocks at the interior origins
      for (int i = 0; i < 2; ++i) for (int j = 0; j < 2; ++j) {
        acc_buf(pl.xs[l], nb, b, i + pl.xs[l].prow, j + pl.xs[l].pcol, WF, "tiny-x");
        acc_buf(pl.ds[l], nb, b, i + pl.ds[l].prow, j + pl.ds[l].pcol, WF, "tiny-d");
      }
    } else {
      // x bands: pcol 0, reads left of a row's interior land in the previous
      // row's right margin or in the 4 floats ahead of the buffer
      const WtBuf X = pl.xs[l];
      CHECK(X.pcol == 0 && X.prow == R && X.off % 4 == 0 && X.stride >= TCW * pl.tc[l] + R, "x band margins");
      CHECK(((X.off + (long)b * X.band + (long)p0 * X.stride + q0 + X.pcol - 4) % 4) == 0, "corr-x align");
      for (int a = 0; a < TBR + K - 1; ++a) for (int c = 0; c < TCW + K - 1; ++c) {
        const int p = p0 + a - R, q = q0 + c - R;
        const long k = X.off + (long)b * X.band + (long)(p + X.prow) * X.stride + q + X.pcol;
        CHECK(k >= X.off - 4 && k < X.off + 4L * X.band && k >= 0 && k < WF, "corr-x outside x region");
        const bool inside = p >= 0 && p < pl.Hs[l] && q >= 0 && q < pl.Ws[l];
        bool interior = false;
        if (k >= X.off) {  // decode: an interior position of some band of level l?
          const long rel = k - X.off, bi = rel / X.band, r = (rel % X.band) / X.stride - X.prow, cc = (rel % X.band) % X.stride - X.pcol;
          interior = r >= 0 && r < pl.Hs[l] && cc >= 0 && cc < pl.Ws[l];
          if (inside) CHECK(bi == b && r == p && cc == q, "corr-x maps interior wrong");
        }
        if (!inside) CHECK(!interior, "corr-x margin (%d,%d) l=%d is an interior", p, q, l);
      }
      for (int o = 0; o < TBR; ++o) for (int c = 0; c < TCW; ++c) acc_buf(pl.ds[l], nb, b, p0 + o, q0 + c, WF, "corr-d");
    }
    if (l == 0) CHECK(((pl.xs[l].off + p0 * pl.xs[l].stride + q0) % 4) == 0, "corr-x align");
    CHECK(((pl.ds[l].off + p0 * pl.ds[l].stride + q0) % 4) == 0, "corr-d align");
  }
  for (int B = 0; B < pl.nbands; ++B) {
    const int l = B == 0 ? 0 : 1 + (B - 1) / 4, b = B == 0 ? 0 : (B - 1) % 4;
    const int tiles = pl.tr[l] * pl.tc[l];
    CHECK(pl.item_begin[l] + b * tiles + tiles <= pl.items_per_plane, "band item range");
  }
  {
    const long long U = (long long)C * pl.batches;
    CHECK(pl.batches * pl.P >= N && (pl.batches - 1) * pl.P < N, "batches");
    CHECK(pl.grid >= 1 && pl.grid <= U, "grid %d U %lld", pl.grid, U);
    for (int i = 0; i <= pl.grid; ++i) CHECK(bw_unit_begin(pl, i) == (int)(U * i / pl.grid), "unit_begin formula at %d", i);
    std::vector<int> cover(U, 0);
    for (int i = 0; i < pl.grid; ++i) {
      const int ub = bw_unit_begin(pl, i), ue = bw_unit_begin(pl, i + 1);
      CHECK(ub < ue, "empty CTA range");
      for (int u = ub; u < ue; ++u) {
        cover[u]++;
        CHECK(u / pl.batches - ub / pl.batches < pl.nrec, "record slot beyond nrec");
      }
    }
    for (long long u = 0; u < U; ++u) CHECK(cover[u] == 1, "unit %lld covered %d times", u, cover[u]);
    // finalize's CTA search per channel
    for (int c = 0; c < C; ++c) {
      const int G = pl.grid, NB = pl.batches;
      int i0 = (int)((long long)c * NB * G / U);
      while (i0 > 0 && bw_unit_begin(pl, i0) > c * NB) --i0;
      while (bw_unit_begin(pl, i0 + 1) <= c * NB) ++i0;
      int i1 = (int)((long long)(c + 1) * NB * G / U);
      if (i1 < i0 + 1) i1 = i0 + 1;
      while (i1 > i0 + 1 && bw_unit_begin(pl, i1 - 1) >= (c + 1) * NB) --i1;
      while (i1 < G && bw_unit_begin(pl, i1) < (c + 1) * NB) ++i1;
      int units = 0;
      for (int i = i0; i < i1; ++i) {
        const int ub = bw_unit_begin(pl, i), ue = bw_unit_begin(pl, i + 1);
        const int lo = ub > c * NB ? ub : c * NB, hi = ue < (c + 1) * NB ? ue : (c + 1) * NB;
        CHECK(hi > lo, "finalize visits a CTA without units of channel %d", c);
        units += hi - lo;
        CHECK(c - ub / NB >= 0 && c - ub / NB < pl.nrec, "finalize record slot");
      }
      CHECK(units == NB, "finalize covers %d of %d units of channel %d", units, NB, c);
    }
  }
}


static long win_plans = 0, win_unsup = 0;
static void check_win(int N, int C, int H, int W, int L, int K, int mode, int dtype) {
  wtconv_desc_t d{N, C, H, W, L, K, dtype};
  WtFwdPlan pl;
  if (plan_win(&d, pl, mode) != WTCONV_OK) { ++win_unsup; return; }
  ++win_plans;
  const int R = K / 2, TP = pl.ftp, TQ = WT_TQ, ZT = WT_ZT, PF = pl.wf, XF = pl.xf, h = pl.halo;
  const int Hv = pl.Hs[0], Wv = pl.Ws[0], th = pl.th, tw = pl.tw, P = pl.P, S = 1 << L;
  const int A = S > 8 ? S : 8;
  CHECK(pl.win == 1 && pl.win_load == mode, "mode");
  CHECK(th % A == 0 && tw % A == 0 && th > 0 && tw > 0, "tile align th=%d tw=%d", th, tw);
  CHECK(h % 8 == 0 && h % S == 0 && h >= R * S, "halo %d", h);
  CHECK(Hv == th + 2 * h && Wv == tw + 2 * h, "window dims");
  for (int l = 1; l <= L; ++l) CHECK(pl.Hs[l] == Hv >> l && (Hv >> l) << l == Hv && pl.zo[l] == h >> l && (pl.zo[l] << l) == h, "level sizes");
  CHECK(pl.xslot % 32 == 0 && P * XF <= pl.xslot && pl.stage_off == pl.nsets * pl.xslot && pl.stage_off % 32 == 0, "sets");
  CHECK(pl.work_off % 32 == 0 && pl.work_off >= pl.stage_off + (mode == 2 ? (P * Hv * Wv + 1) / 2 : 0), "staging");
  CHECK(pl.work_off + P * PF <= pl.w_off && pl.w_off % 4 == 0 && PF % 4 == 0 && XF % 4 == 0, "work");
  CHECK(pl.mb_off % 2 == 0 && pl.mb_off >= pl.w_off + (1 + 4 * L) * pl.w_band && 4 * pl.mb_off + 16 <= pl.smem_bytes - WT_SMEM_SLACK, "mbar");
  CHECK(pl.smem_bytes <= 232448, "smem");
  CHECK(pl.nsets == 1 || mode == 1, "two sets only for float32 boxes");
  CHECK(pl.lev[0].off == 0 && XF == pl.lev[0].band && pl.lev[0].pcol == 4 && pl.lev[0].prow == R && pl.lev[0].stride == Wv + 8, "x buffer");
  CHECK((long)pl.nty * th >= H && (long)pl.ntx * tw >= W && (long)(pl.nty - 1) * th < H && (long)(pl.ntx - 1) * tw < W, "tile cover");
  CHECK((long)pl.groups * P >= N && (long)(pl.groups - 1) * P < N, "groups");
  CHECK(pl.ftr * TP * 2 == th && pl.ftc * TQ * 2 == tw, "final tile grid");
  if (mode == 1) {
    CHECK(pl.lev[0].stride <= 256 && XF / pl.lev[0].stride <= 256 && pl.lev[0].stride % 4 == 0 && pl.tma_bytes == 4u * P * XF, "box32");
  } else if (mode == 2) {
    CHECK(Wv <= 256 && Hv <= 256 && Wv % 8 == 0 && pl.tma_bytes == 2u * P * Hv * Wv, "box16");
  }
  for (int tx = 0; tx < pl.ntx; ++tx) {
    const int ox = tx * tw - h;
    if (mode == 1) CHECK(((ox - 4) % 4 + 4) % 4 == 0, "box32 x coordinate %d", ox - 4);
    if (mode == 2) CHECK((ox % 8 + 8) % 8 == 0, "box16 x coordinate %d", ox);
    CHECK((ox % 8 + 8) % 8 == 0, "vector load x origin");
  }
  CHECK(Wv % 8 == 0, "window width");
  // one window (plane slot 0; slot g is g*XF / g*PF further, inside the checked regions)
  std::vector<char> xw(XF, 0), pw(PF, 0);
  auto idx = [](const WtBuf& b, int bi, int r, int c) { return (long)b.off + (long)bi * b.band + (long)r * b.stride + c; };
  for (int i = 0; i < Hv; ++i) for (int j = 0; j < Wv; ++j) { acc_buf(pl.lev[0], 1, 0, i + R, j + 4, XF, "wload"); xw[idx(pl.lev[0], 0, i + R, j + 4)] = 1; }
  if (mode == 2) for (int g = 0; g < P; ++g) CHECK(((long)g * Hv * Wv * 2) % 8 == 0 && (long)P * Hv * Wv * 2 <= 4L * (pl.work_off - pl.stage_off), "widen staging");
  auto wrp = [&](const WtBuf& b, int bi, int r, int c, const char* what) { acc_buf(b, 4, bi, r, c, PF, what); long k = idx(b, bi, r, c); if (k >= 0 && k < PF) pw[k] = 1; };
  auto interior = [&](const WtBuf& b, int l, int bi, int p, int q, const char* what) {  // read of level-l position (p, q)
    CHECK(p >= 0 && p < pl.Hs[l] && q >= 0 && q < pl.Ws[l], "%s outside level %d interior (%d,%d)", what, l, p, q);
    acc_buf(b, 4, bi, p + b.prow, q + b.pcol, PF, what);
    long k = idx(b, bi, p + b.prow, q + b.pcol);
    if (k >= 0 && k < PF) CHECK(pw[k], "%s reads unwritten (%d,%d) l=%d", what, p, q, l);
  };
  if (L == 1) {
    for (int p = 0; p < pl.Hs[1]; ++p) for (int q = 0; q < pl.Ws[1]; ++q) {
      for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) CHECK(xw[idx(pl.lev[0], 0, 2 * p + u + R, 2 * q + v + 4)], "wana1 read");
      for (int b = 0; b < 4; ++b) wrp(pl.lev[1], b, p + pl.lev[1].prow, q + pl.lev[1].pcol, "wana1 write");
    }
  } else {
    const WtBuf D1 = pl.lev[1], D2 = pl.lev[2];
    for (int P2 = 0; P2 < pl.Hs[2]; ++P2) for (int Q2 = 0; Q2 < pl.Ws[2]; ++Q2) {
      for (int a = 0; a < 4; ++a) for (int e = 0; e < 4; ++e) CHECK(xw[idx(pl.lev[0], 0, 4 * P2 + a + R, 4 * Q2 + e + 4)], "wana12 read");
      for (int u = 0; u < 2; ++u) {
        const int p = 2 * P2 + u, q = 2 * Q2;
        if (p < pl.Hs[1]) {
          if (q + 1 < pl.Ws[1] && (D1.pcol & 1) == 0) CHECK(idx(D1, 0, p + D1.prow, q + D1.pcol) % 2 == 0, "float2 store align");
          for (int v = 0; v < 2; ++v) if (q + v < pl.Ws[1]) for (int b = 0; b < 4; ++b) wrp(D1, b, p + D1.prow, q + v + D1.pcol, "wana12 w1");
        }
      }
      for (int b = 0; b < 4; ++b) wrp(D2, b, P2 + D2.prow, Q2 + D2.pcol, "wana12 w2");
    }
  }
  for (int l = 3; l <= L; ++l) {
    const WtBuf Sb = pl.lev[l - 1], D = pl.lev[l];
    for (int p = 0; p < pl.Hs[l]; ++p) for (int q = 0; q < pl.Ws[l]; ++q) {
      for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) interior(Sb, l - 1, 0, 2 * p + u, 2 * q + v, "wana read");
      for (int b = 0; b < 4; ++b) wrp(D, b, p + D.prow, q + D.pcol, "wana write");
    }
  }
  const int NV = (ZT + K - 1 + 3) / 4;
  for (int l = 1; l <= L; ++l) {
    const WtBuf Y = pl.lev[l], Z = pl.zb[l];
    const int zo = pl.zo[l], Tl = th >> l, Ul = tw >> l;
    CHECK(Z.off % 4 == 0 && Z.stride % 4 == 0 && Z.band % 4 == 0 && Y.off % 4 == 0 && Y.stride % 4 == 0 && Y.band % 4 == 0, "level buffer align");
    CHECK(pl.ztr[l] * ZT >= Tl && pl.ztc[l] * ZT >= Ul, "z tiles cover");
    for (int b = 0; b < 4; ++b) for (int tp = 0; tp < pl.ztr[l]; ++tp) for (int tq = 0; tq < pl.ztc[l]; ++tq) {
      const int p0 = tp * ZT, q0 = tq * ZT;
      const int r0 = zo + p0 - R + Y.prow, c0 = zo + q0 - R + Y.pcol;
      CHECK(r0 >= 0 && c0 >= 0 && c0 % 4 == 0 && idx(Y, b, r0, c0) % 4 == 0, "zconv window align r0=%d c0=%d", r0, c0);
      for (int a = 0; a < ZT + K - 1; ++a) for (int c = 0; c < 4 * NV; ++c) acc_buf(Y, 4, b, r0 + a, c0 + c, PF, "wzconv read");
      for (int o = 0; o < ZT; ++o) for (int j = 0; j < ZT; ++j) {
        if (!(p0 + o < Tl && q0 + j < Ul)) continue;
        for (int du = 0; du < K; ++du) for (int dv = 0; dv < K; ++dv) interior(Y, l, b, zo + p0 + o - R + du, zo + q0 + j - R + dv, "wzconv tap");
        wrp(Z, b, p0 + o, q0 + j, "wzconv write");
      }
      if (p0 + ZT <= Tl && q0 + ZT <= Ul) for (int o = 0; o < ZT; ++o) CHECK(idx(Z, b, p0 + o, q0) % 4 == 0, "z float4 store");
    }
  }
  auto zread = [&](int l, int b, int p, int q, const char* what) {
    const WtBuf Z = pl.zb[l];
    acc_buf(Z, 4, b, p, q, PF, what);
    long k = idx(Z, b, p, q);
    if (k >= 0 && k < PF) CHECK(pw[k], "%s reads unwritten Z l=%d (%d,%d)", what, l, p, q);
  };
  const int OFF = 4 - R;
  for (int tp = 0; tp < pl.ftr; ++tp) for (int tq = 0; tq < pl.ftc; ++tq) {
    const int p0 = tp * TP, q0 = tq * TQ;
    if (L >= 2) for (int b = 0; b < 4; ++b) for (int k = 0; k < TP / 2; ++k) zread(2, b, (p0 >> 1) + k, q0 >> 1, "wf z2");
    for (int l = 3; l <= L; ++l) for (int b = 0; b < 4; ++b) zread(l, b, p0 >> (l - 1), q0 >> (l - 1), "wf zl");
    for (int o = 0; o < TP; ++o) for (int b = 0; b < 4; ++b) {
      CHECK(idx(pl.zb[1], b, p0 + o, q0) % 2 == 0, "z1 float2 read");
      for (int j = 0; j < TQ; ++j) zread(1, b, p0 + o, q0 + j, "wf z1");
    }
    CHECK((h + 2 * q0) % 4 == 0, "base conv row start");
    for (int a = 0; a < 2 * TP + K - 1; ++a) for (int c = 0; c < 2 * TQ + K - 1; ++c) {
      const int br = h + 2 * p0 + a, bc = h + 2 * q0 + OFF + c;
      acc_buf(pl.lev[0], 1, 0, br, bc, XF, "wf base");
      CHECK(br - R >= 0 && br - R < Hv && bc - 4 >= 0 && bc - 4 < Wv, "base tap outside window (%d,%d)", br - R, bc - 4);
    }
  }
  // global stores and output coverage (small planes: every output written exactly once)
  const bool count = (long)H * W <= 300000;
  std::vector<unsigned char> hits(count ? (size_t)H * W : 0, 0);
  for (int ty = 0; ty < pl.nty; ++ty) for (int tx = 0; tx < pl.ntx; ++tx)
    for (int tp = 0; tp < pl.ftr; ++tp) for (int tq = 0; tq < pl.ftc; ++tq) {
      const int gi0 = ty * th, j0 = tx * tw + 2 * tq * TQ;
      CHECK(j0 % (2 * TQ) == 0, "store column multiple");
      for (int oo = 0; oo < 2 * TP; ++oo) {
        const int i = gi0 + 2 * tp * TP + oo;
        if (i >= H) continue;
        for (int es = 2; es <= 4; es += 2) {
          const bool vec = (W % (16 / es)) == 0;
          if (vec && j0 + 2 * TQ <= W) CHECK((((long)i * W + j0) * es) % (2 * TQ * es) == 0, "vector store align");
        }
        if (count) for (int jj = 0; jj < 2 * TQ; ++jj) if (j0 + jj < W) hits[(size_t)i * W + j0 + jj]++;
      }
    }
  if (count) for (size_t k = 0; k < hits.size(); ++k) CHECK(hits[k] == 1, "output %zu written %d times", k, hits[k]);
}

static void check_grid(const WtBwPlan& pl, int C) {
  const long long U = (long long)C * pl.batches;
  CHECK(pl.grid >= 1 && pl.grid <= U, "grid %d U %lld", pl.grid, U);
  for (int i = 0; i <= pl.grid; ++i) CHECK(bw_unit_begin(pl, i) == (int)(U * i / pl.grid), "unit_begin formula at %d", i);
  if (U > 2000000) return;
  std::vector<int> cover(U, 0);
  for (int i = 0; i < pl.grid; ++i) {
    const int ub = bw_unit_begin(pl, i), ue = bw_unit_begin(pl, i + 1);
    CHECK(ub < ue, "empty CTA range");
    for (int u = ub; u < ue; ++u) { cover[u]++; CHECK(u / pl.batches - ub / pl.batches < pl.nrec, "record slot beyond nrec"); }
  }
  for (long long u = 0; u < U; ++u) CHECK(cover[u] == 1, "unit %lld covered %d times", u, cover[u]);
  for (int c = 0; c < C; ++c) {
    const int G = pl.grid, NB = pl.batches;
    int i0 = (int)((long long)c * G / C);
    while (i0 > 0 && bw_unit_begin(pl, i0) > c * NB) --i0;
    while (bw_unit_begin(pl, i0 + 1) <= c * NB) ++i0;
    int i1 = (int)((long long)(c + 1) * G / C);
    if (i1 < i0 + 1) i1 = i0 + 1;
    while (i1 > i0 + 1 && bw_unit_begin(pl, i1 - 1) >= (c + 1) * NB) --i1;
    while (i1 < G && bw_unit_begin(pl, i1) < (c + 1) * NB) ++i1;
    int units = 0;
    for (int i = i0; i < i1; ++i) {
      const int ub = bw_unit_begin(pl, i), ue = bw_unit_begin(pl, i + 1);
      const int lo = ub > c * NB ? ub : c * NB, hi = ue < (c + 1) * NB ? ue : (c + 1) * NB;
      CHECK(hi > lo, "finalize visits a CTA without units of channel %d", c);
      units += hi - lo;
      CHECK(c - ub / NB >= 0 && c - ub / NB < pl.nrec, "finalize record slot");
    }
    CHECK(units == NB, "finalize covers %d of %d units of channel %d", units, NB, c);
  }
}

static long bww_plans = 0, bww_unsup = 0;
static void check_bw_win(int N, int C, int H, int W, int L, int K, int mode, int dtype) {
  wtconv_desc_t d{N, C, H, W, L, K, dtype};
  WtBwPlan pl;
  if (plan_bw_win(&d, pl, mode) != WTCONV_OK) { ++bww_unsup; return; }
  ++bww_plans;
  const int R = K / 2, KK = K * K, h = pl.halo, Hv = pl.Hs[0], Wv = pl.Ws[0], th = pl.th, tw = pl.tw, P = pl.P;
  const int TR = pl.tbr, S = 1 << L, A = S > 8 ? S : 8, WF = pl.wf, XBF = pl.xbf, DBF = pl.dbf;
  CHECK(TR == 8 || TR == 4, "tbr");
  CHECK(th % A == 0 && tw % A == 0 && h % 8 == 0 && h % S == 0 && h >= R * S, "tile/halo");
  CHECK(Hv == th + 2 * h && Wv == tw + 2 * h, "window");
  for (int l = 0; l <= L; ++l) CHECK(pl.Hs[l] == Hv >> l && pl.dHs[l] == th >> l && pl.dWs[l] == tw >> l && ((pl.dHs[l] << l) == th), "level sizes");
  CHECK(pl.xr % 32 == 0 && pl.xr >= P * XBF && pl.islot % 32 == 0 && pl.islot - pl.xr >= P * DBF, "input set");
  CHECK(pl.stage_off == pl.nsets * pl.islot && pl.stage_off % 32 == 0, "stage off");
  if (mode == 2) CHECK(pl.stage_dx % 32 == 0 && 2L * pl.stage_dx >= (long)P * Hv * Wv && pl.work_off - pl.stage_off - pl.stage_dx >= (P * th * tw + 1) / 2, "staging");
  CHECK(pl.work_off % 4 == 0 && pl.red_floats >= P * WF && pl.red_floats >= P * pl.items_per_plane * (KK + 1), "work");
  CHECK(pl.mb_off % 2 == 0 && pl.mb_off >= pl.work_off + pl.red_floats && 4 * pl.mb_off + 16 + WT_SMEM_SLACK <= pl.smem_bytes && pl.smem_bytes <= 232448, "smem");
  CHECK(pl.nsets == 1 || mode == 1, "two sets only for float32 boxes");
  CHECK(P * pl.items_per_plane <= (TR == 8 ? 1 : 2) * 256, "items per CTA");
  CHECK(pl.xs[0].off == 0 && XBF == pl.xs[0].band && pl.xs[0].pcol == 4 && pl.xs[0].prow == R && pl.xs[0].stride == Wv + 8, "x buffer");
  CHECK(pl.ds[0].off == 0 && DBF == th * tw && pl.ds[0].stride == tw && pl.ds[0].prow == 0 && pl.ds[0].pcol == 0, "dy buffer");
  CHECK((long)pl.nty * th >= H && (long)pl.ntx * tw >= W && (long)(pl.nty - 1) * th < H && (long)(pl.ntx - 1) * tw < W, "tile cover");
  CHECK((long)pl.groups * P >= N && (long)(pl.groups - 1) * P < N && pl.batches == pl.groups * pl.nty * pl.ntx, "groups");
  CHECK(pl.nbands == 1 + 4 * L && pl.part_stride == pl.nbands * (KK + 1), "bands");
  if (mode == 1) CHECK(pl.xs[0].stride <= 256 && XBF / pl.xs[0].stride <= 256 && tw <= 256 && th <= 256 && pl.tma_bytes == 4u * P * (XBF + DBF), "box32");
  if (mode == 2) CHECK(Wv <= 256 && Hv <= 256 && Wv % 8 == 0 && tw % 8 == 0 && pl.tma_bytes == 2u * P * (Hv * Wv + th * tw), "box16");
  for (int tx = 0; tx < pl.ntx; ++tx) {
    const int tx0 = tx * tw;
    CHECK(tx0 % 8 == 0 && ((tx0 - h - 4) % 4 + 4) % 4 == 0 && ((tx0 - h) % 8 + 8) % 8 == 0, "box x coordinates");
  }
  // one unit (plane slot 0)
  std::vector<char> xw(XBF, 0), dw(DBF, 0), pw(WF, 0);
  auto idx = [](const WtBuf& b, int bi, int r, int c) { return (long)b.off + (long)bi * b.band + (long)r * b.stride + c; };
  for (int i = 0; i < Hv; ++i) for (int j = 0; j < Wv; ++j) { acc_buf(pl.xs[0], 1, 0, i + R, j + 4, XBF, "bwx load"); xw[idx(pl.xs[0], 0, i + R, j + 4)] = 1; }
  for (int i = 0; i < th; ++i) for (int j = 0; j < tw; ++j) { acc_buf(pl.ds[0], 1, 0, i, j, DBF, "bwd load"); dw[idx(pl.ds[0], 0, i, j)] = 1; }
  auto wrp = [&](const WtBuf& b, int bi, int r, int c, const char* what) { acc_buf(b, 4, bi, r, c, WF, what); long k = idx(b, bi, r, c); if (k >= 0 && k < WF) pw[k] = 1; };
  auto rdp = [&](const WtBuf& b, int bi, int r, int c, const char* what) { acc_buf(b, 4, bi, r, c, WF, what); long k = idx(b, bi, r, c); if (k >= 0 && k < WF) CHECK(pw[k], "%s reads unwritten", what); };
  // pyramids: x window (xs) and dy tile (ds)
  for (int which = 0; which < 2; ++which) {
    const WtBuf* B = which == 0 ? pl.xs : pl.ds;
    const int* Hs = which == 0 ? pl.Hs : pl.dHs;
    const int* Ws = which == 0 ? pl.Ws : pl.dWs;
    std::vector<char>& in = which == 0 ? xw : dw;
    if (L == 1) {
      for (int p = 0; p < Hs[1]; ++p) for (int q = 0; q < Ws[1]; ++q) {
        for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) CHECK(in[idx(B[0], 0, 2 * p + u + B[0].prow, 2 * q + v + B[0].pcol)], "ana1 read");
        for (int b = 0; b < 4; ++b) wrp(B[1], b, p + B[1].prow, q + B[1].pcol, "ana1 write");
      }
    } else {
      for (int P2 = 0; P2 < Hs[2]; ++P2) for (int Q2 = 0; Q2 < Ws[2]; ++Q2) {
        for (int a = 0; a < 4; ++a) for (int e = 0; e < 4; ++e) CHECK(in[idx(B[0], 0, 4 * P2 + a + B[0].prow, 4 * Q2 + e + B[0].pcol)], "ana12 read");
        if ((B[0].pcol & 3) == 0) for (int a = 0; a < 4; ++a) CHECK(idx(B[0], 0, 4 * P2 + a + B[0].prow, 4 * Q2 + B[0].pcol) % 4 == 0, "ana12 float4 read");
        for (int u = 0; u < 2; ++u) {
          const int p = 2 * P2 + u, q = 2 * Q2;
          if (p < Hs[1]) {
            if (q + 1 < Ws[1] && (B[1].pcol & 1) == 0) CHECK(idx(B[1], 0, p + B[1].prow, q + B[1].pcol) % 2 == 0, "float2 store");
            for (int v = 0; v < 2; ++v) if (q + v < Ws[1]) for (int b = 0; b < 4; ++b) wrp(B[1], b, p + B[1].prow, q + v + B[1].pcol, "ana12 w1");
          }
        }
        for (int b = 0; b < 4; ++b) wrp(B[2], b, P2 + B[2].prow, Q2 + B[2].pcol, "ana12 w2");
      }
    }
    for (int l = 3; l <= L; ++l)
      for (int p = 0; p < Hs[l]; ++p) for (int q = 0; q < Ws[l]; ++q) {
        for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) rdp(B[l - 1], 0, 2 * p + u + B[l - 1].prow, 2 * q + v + B[l - 1].pcol, "ana read");
        for (int b = 0; b < 4; ++b) wrp(B[l], b, p + B[l].prow, q + B[l].pcol, "ana write");
      }
  }
  // correlations
  CHECK(pl.zo[0] == h, "level-0 tile origin");
  for (int l = 0; l <= L; ++l) {
    const WtBuf Xb = pl.xs[l], Db = pl.ds[l];
    const int nb = l == 0 ? 1 : 4;
    CHECK(Xb.stride % 4 == 0 && Db.stride % 4 == 0 && Xb.off % 4 == 0 && Db.off % 4 == 0 && Xb.band % 4 == 0 && Db.band % 4 == 0, "corr buffers align");
    CHECK(pl.tr[l] * TR >= pl.dHs[l] && pl.tc[l] * 4 >= pl.dWs[l], "corr tiles cover");
    for (int b = 0; b < nb; ++b) for (int tp = 0; tp < pl.tr[l]; ++tp) for (int tq = 0; tq < pl.tc[l]; ++tq) {
      const int p0 = tp * TR, q0 = tq * 4;
      // dy rows: lds_row<1> float4 at (p0 + o, q0)
      for (int o = 0; o < TR; ++o) {
        if (l == 0) { acc_buf(Db, 1, 0, p0 + o, q0, DBF, "corr d0"); CHECK(idx(Db, 0, p0 + o, q0) % 4 == 0, "d0 float4"); for (int j = 0; j < 4; ++j) CHECK(p0 + o < th && q0 + j < tw && dw[idx(Db, 0, p0 + o, q0 + j)], "d0 read unloaded"); }
        else { for (int j = 0; j < 4; ++j) acc_buf(Db, 4, b, p0 + o, q0 + j, WF, "corr dl"); CHECK(idx(Db, b, p0 + o, q0) % 4 == 0, "dl float4");
               for (int j = 0; j < 4; ++j) { long k = idx(Db, b, p0 + o, q0 + j); if (p0 + o < pl.dHs[l] && q0 + j < pl.dWs[l]) CHECK(pw[k], "dl real position unwritten"); else CHECK(!pw[k], "dl margin written (not zero)"); } }
      }
      if (l == 0) {
        const int r0 = h + p0, c0 = h + q0;  // buffer row/col of the aligned window base; OFF = 4 - R
        CHECK(c0 % 4 == 0 && idx(Xb, 0, r0, c0) % 4 == 0, "x0 base align");
        for (int a = 0; a < TR + K - 1; ++a) for (int c = 0; c < 4 + K - 1; ++c) acc_buf(Xb, 1, 0, r0 + a, c0 + 4 - R + c, XBF, "corr x0");
        for (int o = 0; o < TR; ++o) for (int j = 0; j < 4; ++j) for (int du = 0; du < K; ++du) for (int dv = 0; dv < K; ++dv) {
          const int ii = h + p0 + o - R + du, jj = h + q0 + j - R + dv;
          CHECK(ii >= 0 && ii < Hv && jj >= 0 && jj < Wv, "x0 tap outside window");
        }
      } else {
        const int zo = pl.zo[l];
        const int r0 = zo + p0 - R + Xb.prow, c0 = zo + q0 + Xb.pcol - 4;  // aligned base; OFF = 4 - R
        CHECK(r0 >= 0 && c0 >= 0 && c0 % 4 == 0 && idx(Xb, b, r0, c0) % 4 == 0, "xl window align");
        for (int a = 0; a < TR + K - 1; ++a) for (int c = 0; c < 4 + K - 1; ++c) acc_buf(Xb, 4, b, r0 + a, c0 + 4 - R + c, WF, "corr xl");
        for (int o = 0; o < TR; ++o) for (int j = 0; j < 4; ++j) {
          if (!(p0 + o < pl.dHs[l] && q0 + j < pl.dWs[l])) continue;
          for (int du = 0; du < K; ++du) for (int dv = 0; dv < K; ++dv) {
            const int p = zo + p0 + o - R + du, q = zo + q0 + j - R + dv;
            CHECK(p >= 0 && p < pl.Hs[l] && q >= 0 && q < pl.Ws[l], "xl tap outside window level");
            rdp(Xb, b, p + Xb.prow, q + Xb.pcol, "xl tap");
          }
        }
      }
    }
  }
  check_grid(pl, C);
}

static long bwf_plans = 0, bwf_unsup = 0;
static void check_bwf(int N, int C, int H, int W, int L, int K, int dtype) {
  wtconv_desc_t d{N, C, H, W, L, K, dtype};
  WtBwPlan pl; WtFwdPlan fp;
  if (plan_bwf(&d, pl, fp) != WTCONV_OK) { ++bwf_unsup; return; }
  ++bwf_plans;
  const int R = K / 2, KK = K * K, P = pl.P, TR = pl.tbr, TP = fp.ftp, TQ = WT_TQ, ZT = WT_ZT;
  const int XB = pl.xbf, DB = pl.dbf, WF = pl.wf;
  CHECK(TR == 8 && TP == 2, "tiles");
  CHECK(pl.xr % 32 == 0 && pl.xr >= P * XB && pl.islot % 32 == 0 && pl.islot - pl.xr >= P * DB, "input set");
  // 16-bit planes of whole 8-byte chunks are staged raw, unless the staging
  // area would cost the second CTA per SM (then they are loaded element-wise)
  const bool staging = dtype != 0 && (2L * H * W) % 8 == 0 && pl.work_off > pl.stage_off;
  CHECK(pl.stage_off == pl.nsets * pl.islot && pl.stage_off % 32 == 0, "stage off");
  CHECK(pl.work_off == pl.stage_off + (staging ? (P * H * W + 31) / 32 * 32 : 0) && pl.work_off % 4 == 0, "work off");
  if (staging) {
    CHECK(pl.nsets == 1, "staging uses one input set");
    set_bulk(pl, &d, (const void*)(uintptr_t)4096, 4L * (pl.work_off - pl.stage_off) / 2);
    CHECK(pl.use_bulk == 1 || pl.use_bulk == 2, "staging mode");
    CHECK((long)P * H * W * 2 * 2 <= 4L * (pl.work_off - pl.stage_off), "staging capacity");
    const long dyoff = 4L * pl.stage_off + 2L * P * H * W;  // bytes from the (128-byte aligned) base to the raw dy planes
    for (int g = 0; g < P; ++g) {
      const long xo = 4L * pl.stage_off + 2L * g * H * W, dof = dyoff + 2L * g * H * W;
      CHECK(xo % (pl.use_bulk == 1 ? 16 : 8) == 0 && dof % (pl.use_bulk == 1 ? 16 : 8) == 0, "staging plane alignment");
    }
    if (pl.wd_vec == 4) CHECK(W % 4 == 0 && pl.xs[0].pcol % 4 == 0 && pl.ds[0].pcol % 4 == 0, "widen alignment");
    if (pl.wd_vec == 2) CHECK(W % 2 == 0 && pl.xs[0].pcol % 2 == 0 && pl.ds[0].pcol % 2 == 0 && XB % 2 == 0 && DB % 2 == 0, "widen pair alignment");
    if (L >= 2 && W % 4 == 0) {
      check_widen12(H, W, pl.Hs[2], pl.Ws[2], pl.xs[0], XB);
      check_widen12(H, W, pl.Hs[2], pl.Ws[2], pl.ds[0], DB);
    }
    pl.use_bulk = 0;
  } else if (dtype != 0) {
    set_bulk(pl, &d, (const void*)(uintptr_t)4096, 0);
    CHECK(pl.use_bulk == 0, "element-wise loads without a staging area");
  }
  CHECK(pl.red_floats >= P * WF && pl.red_floats >= P * pl.items_per_plane * (KK + 1) && pl.red_floats % 4 == 0, "red");
  CHECK(fp.w_off == pl.work_off + pl.red_floats && fp.w_off % 4 == 0 && fp.w_band % 4 == 0, "weights off");
  CHECK(pl.mb_off % 2 == 0 && pl.mb_off >= fp.w_off + (1 + 4 * L) * fp.w_band && 4 * pl.mb_off + 16 + WT_SMEM_SLACK <= pl.smem_bytes && pl.smem_bytes <= 232448, "smem");
  CHECK(P * pl.items_per_plane <= (TR == 8 ? 1 : 2) * WT_BW_THREADS, "items per CTA");
  CHECK(pl.xs[0].off == 0 && pl.ds[0].off == 0 && XB == pl.xs[0].band && DB == pl.ds[0].band, "plane buffers");
  CHECK(pl.xs[0].pcol == 4 && pl.xs[0].prow == R && pl.ds[0].pcol == 4 && pl.ds[0].prow == R, "plane margins");
  CHECK(pl.xs[0].stride % 4 == 0 && pl.ds[0].stride % 4 == 0, "box inner extent");
  CHECK(pl.tma_bytes == 4u * P * (XB + DB), "tma bytes");
  CHECK(fp.xf == DB && fp.wf == WF && fp.L == L && fp.C == C && fp.H == H && fp.W == W, "fwd view");
  for (int l = 0; l <= L; ++l) CHECK(fp.lev[l].off == pl.ds[l].off && fp.lev[l].stride == pl.ds[l].stride && fp.lev[l].band == pl.ds[l].band && fp.lev[l].prow == pl.ds[l].prow && fp.lev[l].pcol == pl.ds[l].pcol, "fwd view lev");
  for (int l = 1; l <= L; ++l) CHECK(pl.ds[l].pcol == 4 && pl.ds[l].prow == R && pl.xs[l].pcol == 0 && pl.xs[l].prow == R && pl.xs[l].off % 4 == 0, "level margins");
  // shadow: owner tags in the work area (1 x pyramid, 2 dy pyramid, 3 Z) and written flags
  std::vector<char> own(WF, 0), wr(WF, 0), xw(XB, 0), dw(DB, 0);
  auto tag = [&](const WtBuf& b, int nb, int t) { for (long i = b.off; i < b.off + (long)nb * b.band; ++i) { CHECK(i >= 0 && i < WF, "region beyond work area"); if (i >= 0 && i < WF) { CHECK(own[i] == 0, "regions overlap"); own[i] = t; } } };
  for (int l = 1; l <= L; ++l) { tag(pl.xs[l], 4, 1); tag(pl.ds[l], 4, 2); tag(fp.zb[l], 4, 3); }
  auto idx = [](const WtBuf& b, int bi, int r, int c) { return (long)b.off + (long)bi * b.band + (long)r * b.stride + c; };
  for (int i = 0; i < H; ++i) for (int j = 0; j < W; ++j) {
    acc_buf(pl.xs[0], 1, 0, i + R, j + 4, XB, "fx load"); xw[idx(pl.xs[0], 0, i + R, j + 4)] = 1;
    acc_buf(pl.ds[0], 1, 0, i + R, j + 4, DB, "fd load"); dw[idx(pl.ds[0], 0, i + R, j + 4)] = 1;
  }
  // reads of interior position (p, q) of a level-l buffer: written if inside the level, else an unwritten margin
  auto rd = [&](const WtBuf& b, int bi, int l, int p, int q, const char* what, bool workarea, std::vector<char>& flags, int lim) {
    const long k = idx(b, bi, p + b.prow, q + b.pcol);
    CHECK(p + b.prow >= 0 && p + b.prow < b.band / b.stride && q + b.pcol >= 0 && q + b.pcol < b.stride, "%s outside buffer (%d,%d) l=%d", what, p, q, l);
    CHECK(k >= 0 && k < lim, "%s index", what);
    if (k < 0 || k >= lim) return;
    const bool inside = p >= 0 && p < (l == 0 ? H : pl.Hs[l]) && q >= 0 && q < (l == 0 ? W : pl.Ws[l]);
    if (inside) CHECK(flags[k], "%s reads unwritten interior (%d,%d) l=%d", what, p, q, l);
    else CHECK(!flags[k], "%s margin (%d,%d) l=%d was written", what, p, q, l);
  };
  auto wrt = [&](const WtBuf& b, int bi, int p, int q, int want) {
    const long k = idx(b, bi, p + b.prow, q + b.pcol);
    CHECK(k >= 0 && k < WF && own[k] == want, "write outside its region");
    if (k >= 0 && k < WF) wr[k] = 1;
  };
  // pyramids
  for (int sdx = 0; sdx < 2; ++sdx) {
    const WtBuf* B = sdx ? pl.ds : pl.xs;
    std::vector<char>& in = sdx ? dw : xw;
    const int lim0 = sdx ? DB : XB, tg = sdx ? 2 : 1;
    if (L == 1) {
      for (int p = 0; p < pl.Hs[1]; ++p) for (int q = 0; q < pl.Ws[1]; ++q) {
        for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) rd(B[0], 0, 0, 2 * p + u, 2 * q + v, "ana1", false, in, lim0);
        for (int b = 0; b < 4; ++b) wrt(B[1], b, p, q, tg);
      }
    } else {
      for (int P2 = 0; P2 < pl.Hs[2]; ++P2) for (int Q2 = 0; Q2 < pl.Ws[2]; ++Q2) {
        for (int a = 0; a < 4; ++a) { for (int e = 0; e < 4; ++e) rd(B[0], 0, 0, 4 * P2 + a, 4 * Q2 + e, "ana12", false, in, lim0);
          if ((B[0].pcol & 3) == 0) CHECK(idx(B[0], 0, 4 * P2 + a + B[0].prow, 4 * Q2 + B[0].pcol) % 4 == 0, "ana12 float4"); }
        for (int u = 0; u < 2; ++u) {
          const int p = 2 * P2 + u, q = 2 * Q2;
          if (p < pl.Hs[1]) {
            if (q + 1 < pl.Ws[1] && (B[1].pcol & 1) == 0) CHECK(idx(B[1], 0, p + B[1].prow, q + B[1].pcol) % 2 == 0, "float2 store");
            for (int v = 0; v < 2; ++v) if (q + v < pl.Ws[1]) for (int b = 0; b < 4; ++b) wrt(B[1], b, p, q + v, tg);
          }
        }
        for (int b = 0; b < 4; ++b) wrt(B[2], b, P2, Q2, tg);
      }
    }
    for (int l = 3; l <= L; ++l)
      for (int p = 0; p < pl.Hs[l]; ++p) for (int q = 0; q < pl.Ws[l]; ++q) {
        for (int u = 0; u < 2; ++u) for (int v = 0; v < 2; ++v) rd(B[l - 1], 0, l - 1, 2 * p + u, 2 * q + v, "ana", true, wr, WF);
        for (int b = 0; b < 4; ++b) wrt(B[l], b, p, q, tg);
      }
  }
  // correlations
  const int NV = (4 + K - 1 + 3) / 4;
  for (int item = 0; item < pl.items_per_plane; ++item) {
    int l = 0;
    while (l < L && item >= pl.item_begin[l + 1]) ++l;
    const int tiles = pl.tr[l] * pl.tc[l], rel = item - pl.item_begin[l], b = rel / tiles, t = rel - b * tiles, tp = t / pl.tc[l];
    const int p0 = tp * TR, q0 = (t - tp * pl.tc[l]) * 4;
    const WtBuf Xb = pl.xs[l], Db = pl.ds[l];
    CHECK(idx(Db, b, p0 + Db.prow, q0 + Db.pcol) % 4 == 0, "D float4");
    for (int o = 0; o < TR; ++o) for (int j = 0; j < 4; ++j) {
      if (l == 0) rd(Db, 0, 0, p0 + o, q0 + j, "corr d0", false, dw, DB); else rd(Db, b, l, p0 + o, q0 + j, "corr dl", true, wr, WF);
    }
    if (l == 0) {
      CHECK(idx(Xb, 0, p0, q0) % 4 == 0, "x0 align");
      for (int a = 0; a < TR + K - 1; ++a) for (int c = 0; c < 4 + K - 1; ++c) rd(Xb, 0, 0, p0 + a - R, q0 + c - R, "corr x0", false, xw, XB);
    } else {
      CHECK(idx(Xb, b, p0, q0 + Xb.pcol - 4) % 4 == 0, "xl align");
      for (int a = 0; a < TR + K - 1; ++a) for (int c = 0; c < 4 + K - 1; ++c) {
        const int p = p0 + a - R, q = q0 + c - R;
        const long k = idx(Xb, b, p + Xb.prow, q + Xb.pcol);
        CHECK(k >= Xb.off - 4 && k < Xb.off + 4L * Xb.band && k >= 0 && k < WF, "corr xl outside x region");
        if (k < 0 || k >= WF) continue;
        const bool inside = p >= 0 && p < pl.Hs[l] && q >= 0 && q < pl.Ws[l];
        if (inside) CHECK(wr[k] && own[k] == 1, "corr xl unwritten interior");
        else CHECK(!wr[k] && (own[k] == 1 || own[k] == 0), "corr xl margin written (%d,%d) l=%d", p, q, l);
      }
    }
  }
  // band convolutions of the dy pyramid
  const int ZR = WT_ZT;
  for (int l = 1; l <= L; ++l) for (int b = 0; b < 4; ++b) for (int tp = 0; tp < fp.ztr[l]; ++tp) for (int tq = 0; tq < fp.ztc[l]; ++tq) {
    const int p0 = tp * ZR, q0 = tq * ZT;
    const WtBuf Yb = pl.ds[l];
    CHECK(idx(Yb, b, p0 - R + Yb.prow, q0 + Yb.pcol - 4) % 4 == 0, "zconv row0 align");
    for (int a = 0; a < ZR + K - 1; ++a) for (int c = 0; c < ZT + K - 1; ++c) rd(Yb, b, l, p0 - R + a, q0 - R + c, "zconv", true, wr, WF);
  }
  for (int l = 1; l <= L; ++l) CHECK(fp.ztr[l] * ZR >= pl.Hs[l] && fp.ztc[l] * ZT >= pl.Ws[l], "z tiles cover");
  for (int l = 1; l <= L; ++l) for (int b = 0; b < 4; ++b) for (int tp = 0; tp < fp.ztr[l]; ++tp) for (int tq = 0; tq < fp.ztc[l]; ++tq) {
    const int p0 = tp * ZR, q0 = tq * ZT;
    for (int o = 0; o < ZR; ++o) for (int j = 0; j < ZT; ++j) if (p0 + o < pl.Hs[l] && q0 + j < pl.Ws[l]) wrt(fp.zb[l], b, p0 + o, q0 + j, 3);
    if (p0 + ZR <= pl.Hs[l] && q0 + ZT <= pl.Ws[l]) for (int o = 0; o < ZR; ++o) CHECK(idx(fp.zb[l], b, p0 + o, q0) % 4 == 0, "z float4");
  }
  // final tiles (dx)
  for (int tp = 0; tp < fp.ftr; ++tp) for (int tq = 0; tq < fp.ftc; ++tq) {
    const int p0 = tp * TP, q0 = tq * TQ;
    auto zr = [&](int l, int b, int p, int q) { const WtBuf Z = fp.zb[l]; acc_buf(Z, 4, b, p, q, WF, "f z"); const long k = idx(Z, b, p, q);
      if (k >= 0 && k < WF) { CHECK(own[k] == 3, "f z outside Z"); if (p < pl.Hs[l] && q < pl.Ws[l]) CHECK(wr[k], "f z unwritten valid"); } };
    if (L >= 2) for (int b = 0; b < 4; ++b) for (int k2 = 0; k2 < TP / 2; ++k2) zr(2, b, (p0 >> 1) + k2, q0 >> 1);
    for (int l = 3; l <= L; ++l) for (int b = 0; b < 4; ++b) zr(l, b, p0 >> (l - 1), q0 >> (l - 1));
    for (int o = 0; o < TP; ++o) for (int b = 0; b < 4; ++b) { CHECK(idx(fp.zb[1], b, p0 + o, q0) % 2 == 0, "z1 float2"); for (int j = 0; j < TQ; ++j) zr(1, b, p0 + o, q0 + j); }
    CHECK(idx(pl.ds[0], 0, 2 * p0, 2 * q0) % 4 == 0, "base row align");
    for (int a = 0; a < 2 * TP + K - 1; ++a) for (int c = 0; c < 2 * TQ + K - 1; ++c) rd(pl.ds[0], 0, 0, 2 * p0 + a - R, 2 * q0 + c - R, "f base", false, dw, DB);
  }
  CHECK((long)pl.batches * P >= N && (long)(pl.batches - 1) * P < N, "batches");
  check_grid(pl, C);
}

int main(int argc, char** argv) {
  if (argc > 2 && std::string(argv[1]) == "file") {
    // The layers of a test file: each must be accepted by the whole-plane or
    // the windowed plan of every pass, and every plan must replay cleanly.
    FILE* f = fopen(argv[2], "r");
    if (!f) { printf("cannot open %s\n", argv[2]); return 2; }
    int N, C, H, W, L, K, dt, n = 0, refused = 0;
    while (fscanf(f, "%d %d %d %d %d %d %d", &N, &C, &H, &W, &L, &K, &dt) == 7) {
      ++n;
      g_dtype = dt == 0 ? 0 : 1;
      check_fwd(N, C, H, W, L, K);
      check_bw(N, C, H, W, L, K);
      check_bwf(N, C, H, W, L, K, dt);
      // window load mode of a 16-byte aligned buffer: float32 / 16-bit boxes where rows allow, else plain loads
      const int lm = dt == 0 ? (W % 4 == 0 ? 1 : 0) : (W % 8 == 0 ? 2 : 0);
      for (int mode = 0; mode <= lm; mode += (lm ? lm : 1)) {
        check_win(N, C, H, W, L, K, mode, dt);
        check_bw_win(N, C, H, W, L, K, mode, dt);
      }
      wtconv_desc_t d{N, C, H, W, L, K, (wtconv_dtype_t)dt};
      WtFwdPlan fp;
      WtBwPlan bp;
      const bool fok = plan_fwd(&d, fp) == WTCONV_OK || plan_win(&d, fp, lm) == WTCONV_OK;
      const bool bok = plan_bw(&d, bp) == WTCONV_OK || plan_bw_win(&d, bp, lm) == WTCONV_OK;
      if (!fok || !bok) {
        ++refused;
        printf("refused: %d %d %d %d %d %d %d (forward %d, gradient %d)\n", N, C, H, W, L, K, dt, fok, bok);
      }
    }
    fclose(f);
    printf("layers: %d, refused: %d, window plans %ld, window gradient plans %ld, fused plans %ld\n", n, refused,
           win_plans, bww_plans, bwf_plans);
    printf("errors: %ld\n", errors);
    return errors != 0 || refused != 0;
  }
  // Whole-plane forward / input-gradient and parameter-gradient plans.
  const int shapes[][6] = {
      {2, 3, 13, 17, 3, 5}, {1, 2, 9, 7, 2, 3}, {3, 2, 20, 12, 4, 7}, {2, 2, 33, 31, 5, 9}, {1, 1, 1, 1, 1, 3},
      {1, 2, 1, 9, 2, 5}, {2, 3, 7, 7, 5, 5}, {2, 4, 56, 56, 3, 5}, {3, 4, 28, 28, 2, 5}, {5, 4, 14, 14, 3, 5},
      {9, 6, 7, 7, 2, 5}, {2, 2, 40, 40, 1, 5}, {2, 2, 64, 48, 6, 3}, {1, 2, 5, 64, 3, 5}, {37, 3, 7, 7, 4, 3},
      {2, 32, 32, 32, 2, 5}, {64, 96, 56, 56, 3, 5}, {128, 192, 28, 28, 2, 5}, {2, 3, 19, 23, 3, 3},
      {2, 3, 19, 23, 3, 7}, {2, 3, 19, 23, 3, 9}, {2, 3, 21, 18, 3, 5}, {2, 3, 16, 16, 2, 5}, {16, 8, 28, 28, 3, 5},
      {2, 4, 24, 20, 3, 5}, {128, 96, 56, 56, 5, 5}, {128, 768, 7, 7, 5, 5}, {128, 384, 14, 14, 3, 5},
      {3, 12, 56, 56, 1, 5}, {3, 12, 56, 56, 5, 5}, {3, 96, 7, 7, 1, 5}, {3, 48, 14, 14, 5, 5},
      {1, 1, 100, 100, 8, 9}, {1, 1, 128, 128, 3, 5}, {1, 1, 2, 2, 8, 9}, {1, 1, 3, 1, 8, 3},
      {1, 2, 104, 104, 3, 3}, {1, 2, 96, 96, 5, 9}, {1, 2, 100, 100, 8, 3}, {1, 2, 3, 512, 1, 5}, {2, 3, 92, 92, 8, 9},
      {1, 2, 56, 56, 8, 9}, {2, 2, 64, 64, 1, 5}, {1, 3, 3, 256, 3, 5}, {2, 2, 56, 55, 5, 7}, {1, 2, 57, 57, 3, 5},
  };
  for (g_dtype = 0; g_dtype < 2; ++g_dtype)
    for (auto& s : shapes) {
      check_fwd(s[0], s[1], s[2], s[3], s[4], s[5]);
      check_bw(s[0], s[1], s[2], s[3], s[4], s[5]);
    }
  for (g_dtype = 0; g_dtype < 2; ++g_dtype)
    for (int H = 1; H <= 40; ++H)
      for (int W = 1; W <= 40; W += (W < 12 ? 1 : 7))
        for (int L = 1; L <= 8; ++L)
          for (int K = 3; K <= 9; K += 2) {
            check_fwd(3, 2, H, W, L, K);
            check_bw(3, 2, H, W, L, K);
          }
  // Very large batches (tens of GB of activations): unit counts, grid splits
  // and record slots in 32-bit arithmetic.
  for (g_dtype = 0; g_dtype < 2; ++g_dtype) {
    check_fwd(4096, 96, 56, 56, 3, 5);
    check_bw(4096, 96, 56, 56, 3, 5);
    check_fwd(8192, 768, 7, 7, 2, 5);
    check_bw(8192, 768, 7, 7, 2, 5);
  }
  check_win(1024, 96, 224, 224, 3, 5, 1, 0);
  check_win(1024, 96, 224, 224, 3, 5, 2, 1);
  check_bw_win(1024, 96, 224, 224, 3, 5, 1, 0);
  check_bw_win(512, 64, 512, 512, 2, 5, 2, 1);
  check_bwf(4096, 96, 56, 56, 3, 5, 0);
  // Windowed plans: every load mode, level count and k on planes of many shapes.
  {
    const int wsh[][2] = {{1, 1}, {7, 9}, {56, 56}, {64, 64}, {100, 100}, {113, 129}, {128, 128}, {150, 150},
                          {200, 136}, {224, 224}, {257, 31}, {3, 600}, {384, 384}, {512, 512}, {1023, 17}};
    for (auto& p : wsh)
      for (int L = 1; L <= 8; ++L)
        for (int K = 3; K <= 9; K += 2)
          for (int mode = 0; mode <= 2; ++mode) {
            const int dt = mode == 1 ? 0 : (mode == 2 ? 1 : ((p[1] + L) & 1) ? 0 : 2);
            if (mode == 1 && p[1] % 4) continue;
            if (mode == 2 && p[1] % 8) continue;
            for (int N : {1, 3, 9}) check_win(N, 2, p[0], p[1], L, K, mode, dt);
          }
    // the windowed layers of the GPU tests and benchmark suites
    const int ts[][7] = {{2, 3, 150, 150, 3, 5, 1}, {1, 2, 113, 129, 3, 5, 0}, {3, 2, 128, 128, 1, 9, 1},
                         {1, 2, 130, 124, 2, 7, 1}, {1, 2, 144, 136, 4, 3, 1}, {1, 2, 160, 152, 4, 5, 1},
                         {1, 2, 168, 160, 5, 3, 1}, {1, 3, 1023, 17, 2, 5, 0}, {2, 2, 200, 136, 4, 3, 2},
                         {1, 2, 120, 120, 3, 5, 2}, {1, 2, 131, 125, 3, 7, 0}, {1, 2, 256, 256, 2, 9, 2},
                         {1, 2, 136, 128, 3, 5, 0}, {2, 2, 192, 192, 3, 5, 1}, {2, 64, 224, 224, 3, 5, 1},
                         {8, 64, 224, 224, 3, 5, 1}, {1, 2, 224, 224, 4, 5, 1}, {16, 64, 224, 224, 3, 5, 2},
                         {32, 64, 224, 224, 2, 5, 1}, {16, 96, 128, 128, 3, 5, 1}, {4, 32, 512, 512, 2, 5, 2},
                         {16, 64, 224, 224, 4, 5, 1}, {16, 64, 224, 224, 1, 5, 1}};
    for (auto& t : ts) {
      for (int m = 0; m <= t[6]; ++m) check_win(t[0], t[1], t[2], t[3], t[4], t[5], m, m == 2 ? 1 : 0);
      if (t[6] == 2) {
        check_win(t[0], t[1], t[2], t[3], t[4], t[5], 2, 2);
        check_win(t[0], t[1], t[2], t[3], t[4], t[5], 0, 2);
      }
    }
    printf("window plans checked: %ld (refused: %ld)\n", win_plans, win_unsup);
  }
  {
    const int wsh[][2] = {{1, 1}, {7, 9}, {56, 56}, {64, 64}, {100, 100}, {113, 129}, {128, 128},
                          {150, 150}, {200, 136}, {224, 224}, {257, 31}, {3, 600}, {384, 384}, {1023, 17}};
    for (auto& p : wsh)
      for (int L = 1; L <= 6; ++L)
        for (int K = 3; K <= 9; K += 2)
          for (int mode = 0; mode <= 2; ++mode) {
            const int dt = mode == 1 ? 0 : (mode == 2 ? 1 : ((p[1] + L) & 1) ? 0 : 2);
            for (int N : {1, 3, 9})
              for (int C : {1, 5}) check_bw_win(N, C, p[0], p[1], L, K, mode, dt);
          }
    printf("window gradient plans checked: %ld (refused: %ld)\n", bww_plans, bww_unsup);
  }
  // Fused backward plans: small planes exhaustively, and the benchmark's layers.
  {
    for (int dt = 0; dt < 2; ++dt)
      for (int H = 1; H <= 64; H += (H < 20 ? 1 : 5))
        for (int W = 1; W <= 64; W += (W < 12 ? 1 : 7))
          for (int L = 1; L <= 8; ++L)
            for (int K = 3; K <= 9; K += 2) check_bwf(3, 2, H, W, L, K, dt);
    const int fs[][6] = {{64, 96, 56, 56, 3, 5}, {128, 192, 28, 28, 2, 5}, {128, 96, 56, 56, 5, 5},
                         {128, 384, 14, 14, 3, 5}, {128, 768, 7, 7, 2, 5}, {2, 32, 32, 32, 2, 5}, {37, 3, 7, 7, 4, 3}};
    for (auto& f : fs)
      for (int dt = 0; dt < 2; ++dt) check_bwf(f[0], f[1], f[2], f[3], f[4], f[5], dt);
    printf("fused backward plans checked: %ld (layers it hands to the separate passes: %ld)\n", bwf_plans, bwf_unsup);
  }
  printf("errors: %ld\n", errors);
  return errors != 0;
}
