// C ABI of libwtconv: argument validation, launch planning, dispatch.
// The declarations and the contract of every entry point are in
// include/wtconv.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/wtconv.h"
#include "wtconv_launch.h"
#include "wtconv_plan.h"

namespace {

thread_local char g_last_error[512] = "";

wtconv_status_t fail(wtconv_status_t st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
wtconv_status_t fail(wtconv_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

wtconv_status_t ok() {
  g_last_error[0] = '\0';
  return WTCONV_OK;
}

constexpr int kMaxSmemPerBlock = 232448;  // 227 KiB opt-in shared memory per CTA on sm_103
constexpr int kSmemPerSm = 233472;        // 228 KiB shared memory per SM
constexpr int kNumSms = 152;              // GB300; only a grid-shaping heuristic
constexpr int kStaticSmem = 16;            // static shared memory of the kernels (a flag word)
constexpr int kFwdBudget = 72 * 1024;     // preferred forward CTA footprint (>= 3 CTAs / SM)
constexpr int kBwBudget = 112 * 1024;     // preferred gradient CTA footprint (>= 2 CTAs / SM)

int round_up(int a, int b) { return (a + b - 1) / b * b; }
int ceil_div(int a, int b) { return (a + b - 1) / b; }

WtDiv make_div(int d) {
  uint32_t s = 0;
  while ((1u << s) < (uint32_t)d) ++s;
  WtDiv f;
  f.shift = s;
  f.mul = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << s) - (uint64_t)d)) / (uint64_t)d + 1);
  return f;
}

size_t elem_size(int dtype) { return dtype == WTCONV_F32 ? 4 : 2; }

wtconv_status_t validate_desc(const wtconv_desc_t* d) {
  if (!d) return fail(WTCONV_ERR_INVALID_ARG, "desc is NULL");
  if (d->N < 0 || d->C < 1 || d->H < 1 || d->W < 1)
    return fail(WTCONV_ERR_INVALID_ARG, "bad shape N=%d C=%d H=%d W=%d", d->N, d->C, d->H, d->W);
  if (d->levels < 1 || d->levels > WT_MAXL)
    return fail(WTCONV_ERR_INVALID_ARG, "levels=%d outside [1, %d]", d->levels, WT_MAXL);
  if (d->k < 3 || d->k > 9 || (d->k % 2) == 0)
    return fail(WTCONV_ERR_INVALID_ARG, "k=%d: must be odd and in [3, 9]", d->k);
  if (d->dtype != WTCONV_F32 && d->dtype != WTCONV_F16 && d->dtype != WTCONV_BF16)
    return fail(WTCONV_ERR_INVALID_ARG, "dtype=%d unknown", d->dtype);
  if ((int64_t)d->N * d->C > INT32_MAX / 2 || (int64_t)d->H * d->W > (1 << 24))
    return fail(WTCONV_ERR_UNSUPPORTED, "shape too large for 32-bit plane indexing");
  return WTCONV_OK;
}

void level_sizes(const wtconv_desc_t* d, int* Hs, int* Ws) {
  Hs[0] = d->H;
  Ws[0] = d->W;
  for (int l = 1; l <= d->levels; ++l) {
    Hs[l] = (Hs[l - 1] + 1) / 2;
    Ws[l] = (Ws[l - 1] + 1) / 2;
  }
}

// A row stride of n floats or more that is 4 mod 8: rows 4 apart then start
// 16 banks apart.
int pad48(int n) {
  const int s = round_up(n, 4);
  return s % 8 == 0 ? s + 4 : s;
}

// Places a plane buffer of `nb` bands at `off`; the interior is er x ec with
// prow/pcol zero rows/columns before it and at least as many after it; rows
// are padded to `min_stride` floats and to a multiple of 4.  Returns the next offset.
int place(WtBuf& b, int off, int er, int ec, int prow, int pcol, int nb, int min_stride = 0) {
  b.off = off;
  b.prow = prow;
  b.pcol = pcol;
  b.stride = round_up(ec + 2 * pcol > min_stride ? ec + 2 * pcol : min_stride, 4);
  b.band = (er + 2 * prow) * b.stride;
  return off + nb * b.band;
}

// Bands of at most 2 x 2 coefficients are convolved and correlated from the
// 2 x 2 block at their interior origin (tiny_band_conv / tiny_band_corr), and
// the next level's analysis reads the same block; so their buffers need no
// margin but one zero row and column after the interior: a 2 x 2 block in a
// row of 4 floats.
bool tiny_band(int h, int w) { return h <= 2 && w <= 2; }

int place_tiny(WtBuf& b, int off) { return place(b, off, 2, 2, 0, 0, 4); }

// Buffer geometry of the forward pass for final tiles of tp x WT_TQ level-1
// positions (2tp x 2WT_TQ outputs).
void fwd_geometry(const wtconv_desc_t* d, WtFwdPlan& pl, int tp) {
  const int R = d->k / 2, L = d->levels;
  pl.ftp = tp;
  pl.ftr = ceil_div(pl.Hs[1], tp);
  pl.ftc = ceil_div(pl.Ws[1], WT_TQ);
  // Input plane (own buffer): R zero rows above, a 4-float (16-byte) left
  // margin so its interior rows are 16-byte aligned.  Rows cover the final
  // tiles' windows (2*tp*ftr + 2R) and row length covers their reads.
  pl.xf = round_up(place(pl.lev[0], 0, 2 * tp * pl.ftr, 2 * WT_TQ * pl.ftc, R, 4, 1, 2 * WT_TQ * pl.ftc + 8), 4);
  int off = 0;  // work area: pyramid levels 1..L, then convolved bands
  pl.zbegin[1] = 0;
  for (int l = 1; l <= L; ++l) {
    pl.ztr[l] = ceil_div(pl.Hs[l], WT_ZT);
    pl.ztc[l] = ceil_div(pl.Ws[l], WT_ZT);
    off = tiny_band(pl.Hs[l], pl.Ws[l]) ? place_tiny(pl.lev[l], off)
                                        : place(pl.lev[l], off, WT_ZT * pl.ztr[l], WT_ZT * pl.ztc[l], R, R, 4);
    pl.zbegin[l + 1] = pl.zbegin[l] + 4 * pl.ztr[l] * pl.ztc[l];
  }
  pl.zipp = pl.zbegin[L + 1];
  for (int l = 1; l <= L; ++l) {
    // Z^l: written at the valid positions (p < H_l, q < W_l) only, read by
    // the final tiles at (p >> (l-1), q >> (l-1)) for every level-1 position
    // of the tile grid; rows/columns read but never written stay zero.
    const int fr = ((tp * pl.ftr - 1) >> (l - 1)) + 1, fc = ((WT_TQ * pl.ftc - 1) >> (l - 1)) + 1;
    off = place(pl.zb[l], off, pl.Hs[l] > fr ? pl.Hs[l] : fr, pl.Ws[l] > fc ? pl.Ws[l] : fc, 0, 0, 4);
  }
  pl.wf = round_up(off, 4);
}

// Plans depend only on the layer geometry, the load mode (windowed passes)
// and the device (occupancy), not on the tensors, so successful plans are
// kept: a call with a known layer does not plan again (planning is a few
// microseconds of host time; a layer's fused backward is one launch, so that
// time would otherwise delay it).  Failures are not kept (their message is
// set by planning).
struct PlanKey {
  int v[9];
  bool operator<(const PlanKey& o) const {
    for (int i = 0; i < 9; ++i)
      if (v[i] != o.v[i]) return v[i] < o.v[i];
    return false;
  }
};

PlanKey plan_key(const wtconv_desc_t* d, int extra) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    dev = -1;
  }
  return PlanKey{{dev, d->N, d->C, d->H, d->W, d->levels, d->k, d->dtype, extra}};
}

template <typename T>
class PlanCache {
 public:
  bool get(const PlanKey& k, T* out) {
    std::lock_guard<std::mutex> lock(mu_);
    auto it = m_.find(k);
    if (it == m_.end()) return false;
    *out = it->second;
    return true;
  }
  void put(const PlanKey& k, const T& v) {
    std::lock_guard<std::mutex> lock(mu_);
    if (m_.size() >= 1024) m_.clear();  // bound the memory of long-running processes with many shapes
    m_[k] = v;
  }

 private:
  std::mutex mu_;
  std::map<PlanKey, T> m_;
};

struct BwfPlans {
  WtBwPlan bw;
  WtFwdPlan fwd;
};

wtconv_status_t plan_fwd_compute(const wtconv_desc_t* d, WtFwdPlan& pl);
wtconv_status_t plan_win_compute(const wtconv_desc_t* d, WtFwdPlan& pl, int load);
wtconv_status_t plan_bw_compute(const wtconv_desc_t* d, WtBwPlan& pl);
wtconv_status_t plan_bwf_compute(const wtconv_desc_t* d, WtBwPlan& pl, WtFwdPlan& fp);
wtconv_status_t plan_bw_win_compute(const wtconv_desc_t* d, WtBwPlan& pl, int load);

wtconv_status_t plan_fwd(const wtconv_desc_t* d, WtFwdPlan& pl) {
  static PlanCache<WtFwdPlan> cache;
  const PlanKey k = plan_key(d, -1);
  if (cache.get(k, &pl)) return WTCONV_OK;
  const wtconv_status_t st = plan_fwd_compute(d, pl);
  if (st == WTCONV_OK) cache.put(k, pl);
  return st;
}

wtconv_status_t plan_win(const wtconv_desc_t* d, WtFwdPlan& pl, int load) {
  static PlanCache<WtFwdPlan> cache;
  const PlanKey k = plan_key(d, load);
  if (cache.get(k, &pl)) return WTCONV_OK;
  const wtconv_status_t st = plan_win_compute(d, pl, load);
  if (st == WTCONV_OK) cache.put(k, pl);
  return st;
}

wtconv_status_t plan_bw(const wtconv_desc_t* d, WtBwPlan& pl) {
  static PlanCache<WtBwPlan> cache;
  const PlanKey k = plan_key(d, -1);
  if (cache.get(k, &pl)) return WTCONV_OK;
  const wtconv_status_t st = plan_bw_compute(d, pl);
  if (st == WTCONV_OK) cache.put(k, pl);
  return st;
}

wtconv_status_t plan_bw_win(const wtconv_desc_t* d, WtBwPlan& pl, int load) {
  static PlanCache<WtBwPlan> cache;
  const PlanKey k = plan_key(d, load);
  if (cache.get(k, &pl)) return WTCONV_OK;
  const wtconv_status_t st = plan_bw_win_compute(d, pl, load);
  if (st == WTCONV_OK) cache.put(k, pl);
  return st;
}

// Test hook (wtconv_test_copy_timeout): while it is on, every launch gives
// its bounded copy waits a limit of 2^20 clock cycles and arms each copy
// barrier with 16 bytes more than its copies deliver, so that each wait runs
// out.  Off: 2^31 cycles and no extra bytes.  Applied to the caller's copy of
// a plan just before its launch (cached plans are not touched).
std::mutex g_hook_mu;
bool g_hook_on = false;

template <typename Plan>
void apply_wait_hook(Plan& pl) {
  std::lock_guard<std::mutex> lock(g_hook_mu);
  pl.wait_shift = g_hook_on ? 20 : 31;
  pl.dbg_extra_tx = g_hook_on ? 16u : 0u;
}

wtconv_status_t plan_bwf(const wtconv_desc_t* d, WtBwPlan& pl, WtFwdPlan& fp) {
  static PlanCache<BwfPlans> cache;
  const PlanKey k = plan_key(d, -1);
  BwfPlans b;
  if (cache.get(k, &b)) {
    pl = b.bw;
    fp = b.fwd;
    return WTCONV_OK;
  }
  const wtconv_status_t st = plan_bwf_compute(d, pl, fp);
  if (st == WTCONV_OK) {
    b.bw = pl;
    b.fwd = fp;
    cache.put(k, b);
  }
  return st;
}

// Loop divisors of the analysis, band-convolution and final-tile phases.
void fwd_divs(WtFwdPlan& pl) {
  const int L = pl.L;
  if (L == 1) {
    pl.an_pp[1] = make_div(pl.Hs[1] * pl.Ws[1]);
    pl.an_w[1] = make_div(pl.Ws[1]);
  } else {
    pl.an_pp[2] = make_div(pl.Hs[2] * pl.Ws[2]);
    pl.an_w[2] = make_div(pl.Ws[2]);
  }
  for (int l = 3; l <= L; ++l) {
    pl.an_pp[l] = make_div(pl.Hs[l] * pl.Ws[l]);
    pl.an_w[l] = make_div(pl.Ws[l]);
  }
  pl.z_ipp = make_div(pl.zipp);
  for (int l = 1; l <= L; ++l) {
    pl.z_tiles[l] = make_div(pl.ztr[l] * pl.ztc[l]);
    pl.z_tc[l] = make_div(pl.ztc[l]);
  }
  pl.f_pp = make_div(pl.ftr * pl.ftc);
  pl.f_c = make_div(pl.ftc);
}

wtconv_status_t plan_fwd_compute(const wtconv_desc_t* d, WtFwdPlan& pl) {
  memset(&pl, 0, sizeof(pl));
  pl.N = d->N; pl.C = d->C; pl.H = d->H; pl.W = d->W; pl.L = d->levels; pl.K = d->k;
  const int L = d->levels, KK = d->k * d->k;
  level_sizes(d, pl.Hs, pl.Ws);
  fwd_geometry(d, pl, WT_TP);
  pl.w_band = round_up(KK, 4);
  const int wfloats = (1 + 4 * L) * pl.w_band;
  // Two input sets: float32 planes stream into one while the other is
  // processed.  (16-bit planes, loaded synchronously, measured faster with
  // the same layout too.)
  pl.nsets = 2;
  const long plane_bytes = 4L * (pl.nsets * pl.xf + pl.wf) + 256;
  if (plane_bytes + 4L * wfloats > kMaxSmemPerBlock)
    return fail(WTCONV_ERR_UNSUPPORTED, "plane %dx%d with %d levels needs %ld B of shared memory (max %d)",
                d->H, d->W, L, plane_bytes + 4L * wfloats, kMaxSmemPerBlock);
  // Planes per unit P and final-tile height: the pair with the least modelled
  // time for the layer.  Each phase of a unit costs (rounds of its items over
  // the CTA's threads) x (the latency of one item, in issue slots measured on
  // the stage shapes), plus a fixed cost per unit (barriers, copy wait).  The
  // layer takes ceil(units / resident CTAs) such units, where a unit is P
  // planes of one channel (the last group of a batch partly idle) and the
  // resident CTAs per SM follow from the kernel's registers and the unit's
  // shared memory; a unit's time grows with the CTAs sharing its SM as
  // CTAs^0.3 (fitted to a sweep of forced P on 30 small-plane layers, where
  // 16-bit kernels fit a fourth CTA below 56 KB).  P is bounded by the
  // shared-memory budget of 3 CTAs per SM.  Half-height final tiles never
  // need more shared memory.
  int fit = (int)((kFwdBudget - 4L * wfloats) / plane_bytes);
  if (fit < 1) fit = 1;
  if (d->N > 0 && fit > d->N) fit = d->N;
  int P = 1, tp = WT_TP;
  {
    const int T = WT_FWD_THREADS;
    const long n12 = L >= 2 ? (long)pl.Hs[2] * pl.Ws[2] : (long)pl.Hs[1] * pl.Ws[1];
    // per unit: 400, plus 200 for every level past the second (its own
    // analysis pass behind a CTA barrier)
    const long c12 = 100, c3 = 30, cz = 16L * KK + 130, cunit = 400 + 200L * (L > 2 ? L - 2 : 0);
    const int regs = wt::fwd_regs(d->k, d->dtype);
    const long ctas_r = regs > 0 ? 65536L / (T * (long)round_up(regs, 8)) : 3;
    const long sms = wt::sm_count() > 0 ? wt::sm_count() : 152;
    double best = -1.0;
    for (int q = 1; q <= fit && q <= 64; ++q) {
      const long smem = 4L * (2L * round_up(q * pl.xf, 32) + (long)q * pl.wf + wfloats) + 16 + WT_SMEM_SLACK;
      long ctas = kSmemPerSm / (smem + 1024 + kStaticSmem);
      if (ctas > ctas_r) ctas = ctas_r;
      if (ctas < 1) ctas = 1;
      const long units = (long)d->C * (d->N > 0 ? ceil_div(d->N, q) : 0);
      const double rounds = (double)((units + ctas * sms - 1) / (ctas * sms)) * pow((double)ctas, 0.3);
      for (int t = WT_TP; t >= WT_TP / 2; t /= 2) {
        const long nf = (long)ceil_div(pl.Hs[1], t) * ceil_div(pl.Ws[1], WT_TQ);
        const long cf = 8L * t * KK + (t == WT_TP ? 400 : 300);  // 2t x 2TQ outputs, k*k FMAs each
        long cost = ceil_div((int)(q * n12), T) * c12 + ceil_div((int)(q * pl.zipp), T) * cz +
                    ceil_div((int)(q * nf), T) * cf + cunit;
        for (int l = 3; l <= L; ++l) cost += ceil_div(q * pl.Hs[l] * pl.Ws[l], T) * c3;
        const double total = rounds * cost + 1e-6 * cost / q;  // equal totals (no units): least per plane
        if (best < 0 || total < best * (1 - 1e-9)) {
          best = total;
          P = q;
          tp = t;
        }
      }
    }
  }
  if (tp != WT_TP) fwd_geometry(d, pl, tp);
  pl.P = P;
  pl.groups = d->N > 0 ? ceil_div(d->N, P) : 0;
  pl.xslot = round_up(P * pl.xf, 32);  // 128-byte aligned buffer sets (TMA destinations)
  // One float32 input set when the second would cost a CTA per SM (3 fit by
  // registers): the next unit is then requested as soon as this one is done
  // with its planes, and the other resident CTAs cover the latency.
  // 16-bit planes: the second region holds the raw planes for the bulk
  // copies; it shrinks to just that staging area (one float32 set) on the
  // same condition.
  int region1 = pl.xslot;
  {
    const long two = 4L * (2 * pl.xslot + (long)P * pl.wf + wfloats) + 16 + WT_SMEM_SLACK;
    const long per3 = kSmemPerSm / 3 - 1024 - kStaticSmem;
    const int staging = round_up((P * d->H * d->W + 1) / 2, 32);  // P raw 16-bit planes, in floats
    const int alt = d->dtype == WTCONV_F32 ? 0 : staging;
    if (two > per3 && two - 4L * (pl.xslot - alt) <= per3) {
      pl.nsets = 1;
      region1 = alt;
    }
  }
  pl.stage_off = pl.xslot;
  pl.work_off = pl.xslot + region1;
  pl.w_off = pl.work_off + P * pl.wf;
  pl.mb_off = round_up(pl.w_off + wfloats, 2);
  pl.smem_bytes = 4 * pl.mb_off + 16 + WT_SMEM_SLACK;
  if (pl.smem_bytes > kMaxSmemPerBlock)
    return fail(WTCONV_ERR_UNSUPPORTED, "plane %dx%d with %d levels needs %d B of shared memory (max %d)",
                d->H, d->W, L, pl.smem_bytes, kMaxSmemPerBlock);
  pl.tma_bytes = (uint32_t)(4L * P * pl.xf);
  fwd_divs(pl);
  return WTCONV_OK;
}

// Windowed forward geometry for th x tw output tiles (multiples of
// max(2^L, 8)) and final tiles of tp x WT_TQ level-1 positions; pl.halo set.
// Window: Hv x Wv = (th + 2h) x (tw + 2h) pixels, level l exactly
// (Hv >> l) x (Wv >> l) coefficients.  Input buffer: the window with r zero
// rows above and below and a 4-float margin left and right (the float32 box
// copy fills exactly this).  Level buffers: no top margin (the tile's
// convolution windows start zo - r >= 0 rows into the window), a column
// margin pcol = (r - zo) mod 4 that puts every convolution window's first
// column on a 16-byte boundary, and room for the rows and float4 columns
// the last band-convolution tiles read past the window.  Z buffers hold the
// tile's coefficients only.
void win_geometry(const wtconv_desc_t* d, WtFwdPlan& pl, int th, int tw, int tp) {
  const int R = d->k / 2, L = d->levels, h = pl.halo;
  const int NV = (WT_ZT + d->k - 1 + 3) / 4;  // float4s per row of a band-convolution window
  pl.th = th;
  pl.tw = tw;
  pl.Hs[0] = th + 2 * h;
  pl.Ws[0] = tw + 2 * h;
  for (int l = 1; l <= L; ++l) {
    pl.Hs[l] = pl.Hs[0] >> l;
    pl.Ws[l] = pl.Ws[0] >> l;
  }
  pl.ftp = tp;
  pl.ftr = th / 2 / tp;
  pl.ftc = tw / 2 / WT_TQ;
  pl.xf = place(pl.lev[0], 0, pl.Hs[0], pl.Ws[0], R, 4, 1);
  int off = 0;
  pl.zbegin[1] = 0;
  for (int l = 1; l <= L; ++l) {
    const int zo = h >> l;
    pl.zo[l] = zo;
    pl.ztr[l] = ceil_div(th >> l, WT_ZT);
    pl.ztc[l] = ceil_div(tw >> l, WT_ZT);
    WtBuf& b = pl.lev[l];
    b.off = off;
    b.prow = 0;
    b.pcol = ((R - zo) % 4 + 4) % 4;
    const int rows = std::max(pl.Hs[l], zo + WT_ZT * pl.ztr[l] + R);
    const int cols = std::max(b.pcol + pl.Ws[l], zo + WT_ZT * (pl.ztc[l] - 1) - R + b.pcol + 4 * NV);
    b.stride = round_up(cols, 4);
    b.band = rows * b.stride;
    off += 4 * b.band;
    pl.zbegin[l + 1] = pl.zbegin[l] + 4 * pl.ztr[l] * pl.ztc[l];
  }
  pl.zipp = pl.zbegin[L + 1];
  for (int l = 1; l <= L; ++l) off = place(pl.zb[l], off, th >> l, tw >> l, 0, 0, 4);
  pl.wf = round_up(off, 4);
}

// Shared memory of a windowed plan with P planes per unit and `nsets` input
// sets: [input sets][16-bit staging][P work areas][weights][2 mbarriers].
long win_smem_bytes(const WtFwdPlan& pl, int P, int nsets, int load, int wfloats) {
  const long xslot = round_up(P * pl.xf, 32);
  const long stage = load == 2 ? round_up((P * pl.Hs[0] * pl.Ws[0] + 1) / 2, 32) : 0;
  const long mb = (nsets * xslot + stage + (long)P * pl.wf + wfloats + 1) / 2 * 2;
  return 4 * mb + 16 + WT_SMEM_SLACK;
}

// Windowed plan for planes too large for plan_fwd.  `load`: 0 = plain loads,
// 1 = float32 box copies, 2 = 16-bit box copies (see WtFwdPlan::win_load).
// Tile size, final-tile height, input sets and planes per unit minimise the
// modelled time of the whole call: the phase-round cost of one unit (as in
// plan_fwd, with the pyramid over the whole window) times the number of units
// (edge tiles count whole), weighted by how many CTAs fit an SM: fewer
// resident CTAs hide less latency, which also makes full-height final tiles
// (fewer, longer items) cost more.  The weights were fitted to a sweep of
// forced tilings on a GB300 (224 x 224 planes at levels 1-4 and k = 3, 5, 7;
// 128 x 128 and 512 x 512 planes; float32 and float16), where the model's
// choice came within 2% of the fastest tiling measured.
wtconv_status_t plan_win_compute(const wtconv_desc_t* d, WtFwdPlan& pl, int load) {
  memset(&pl, 0, sizeof(pl));
  pl.N = d->N; pl.C = d->C; pl.H = d->H; pl.W = d->W; pl.L = d->levels; pl.K = d->k;
  const int R = d->k / 2, L = d->levels, KK = d->k * d->k, S = 1 << L;
  pl.win = 1;
  pl.win_load = load;
  pl.halo = round_up(R * S, 8);
  const int h = pl.halo, A = S > 8 ? S : 8;
  pl.w_band = round_up(KK, 4);
  const int wfloats = (1 + 4 * L) * pl.w_band;
  const int thmax = round_up(d->H, A), twmax = round_up(d->W, A);
  const int NT = WT_FWD_THREADS;
  const long c12 = 100, c3 = 30, cz = 16L * KK + 130, cunit = 400 + 200L * (L > 2 ? L - 2 : 0);
  const int Pmax = d->N < 1 ? 1 : (d->N < 8 ? d->N : 8);
  double best = -1.0;
  int bth = 0, btw = 0, btp = 0, bP = 0, bns = 0;
  for (int T = A;; T += A) {
    const int th = T < thmax ? T : thmax, tw = T < twmax ? T : twmax;
    // one box copy per window and plane: at most 256 elements per dimension
    if (tw + 2 * h + 8 > 256 || th + 2 * h + 2 * R > 256) break;
    for (int t = WT_TP; t >= WT_TP / 2; t /= 2) {
      win_geometry(d, pl, th, tw, t);
      const int n12 = L >= 2 ? pl.Hs[2] * pl.Ws[2] : pl.Hs[1] * pl.Ws[1];
      const int nf = pl.ftr * pl.ftc;
      const long cf = 8L * t * KK + (t == WT_TP ? 400 : 300);
      for (int q = 1; q <= Pmax; ++q) {
        for (int ns = (load == 1 ? 2 : 1); ns >= 1; --ns) {
          const long smem = win_smem_bytes(pl, q, ns, load, wfloats);
          if (smem > kMaxSmemPerBlock) continue;
          long ctas = kSmemPerSm / (smem + 1024);
          if (ctas > 3) ctas = 3;
          const long cft = cf + (t == WT_TP ? 150 * (3 - ctas) : 0);
          long cost = ceil_div(q * n12, NT) * c12 + ceil_div(q * pl.zipp, NT) * cz + ceil_div(q * nf, NT) * cft + cunit;
          for (int l = 3; l <= L; ++l) cost += ceil_div(q * pl.Hs[l] * pl.Ws[l], NT) * c3;
          if (load == 0) cost += ceil_div(q * pl.Hs[0] * pl.Ws[0] / 4, NT) * 60;  // plain loads stall the unit
          const double units = (double)ceil_div(d->N > 0 ? d->N : 1, q) * ceil_div(d->H, th) * ceil_div(d->W, tw);
          const double occ = ctas >= 3 ? 1.0 : ctas == 2 ? 1.25 : 2.0;
          const double one_set = (load == 1 && ns == 1) ? 1.05 : 1.0;
          const double total = (double)cost * units * occ * one_set;
          if (best < 0 || total < best * (1 - 1e-9)) {
            best = total;
            bth = th; btw = tw; btp = t; bP = q; bns = ns;
          }
        }
      }
    }
    if (th == thmax && tw == twmax) break;
  }
  if (best < 0)
    return fail(WTCONV_ERR_UNSUPPORTED,
                "plane %dx%d does not fit one CTA, and neither does the smallest %dx%d tile with its %d-pixel halo "
                "(levels %d, k %d)", d->H, d->W, A, A, h, L, d->k);
  win_geometry(d, pl, bth, btw, btp);
  const int P = bP;
  pl.P = P;
  pl.nsets = bns;
  pl.groups = d->N > 0 ? ceil_div(d->N, P) : 0;
  pl.nty = ceil_div(d->H, bth);
  pl.ntx = ceil_div(d->W, btw);
  if ((long long)d->C * pl.groups * pl.nty * pl.ntx >= INT32_MAX)
    return fail(WTCONV_ERR_UNSUPPORTED, "%lld tile units exceed the 32-bit unit index",
                (long long)d->C * pl.groups * pl.nty * pl.ntx);
  pl.xslot = round_up(P * pl.xf, 32);
  const int stage = load == 2 ? round_up((P * pl.Hs[0] * pl.Ws[0] + 1) / 2, 32) : 0;
  pl.stage_off = pl.nsets * pl.xslot;
  pl.work_off = pl.stage_off + stage;
  pl.w_off = pl.work_off + P * pl.wf;
  pl.mb_off = round_up(pl.w_off + wfloats, 2);
  pl.smem_bytes = 4 * pl.mb_off + 16 + WT_SMEM_SLACK;
  pl.tma_bytes = load == 1 ? (uint32_t)(4L * P * pl.xf) : load == 2 ? (uint32_t)(2L * P * pl.Hs[0] * pl.Ws[0]) : 0u;
  pl.wd_vec = 4;
  pl.wd_pp = make_div(pl.Hs[0] * pl.Ws[0] / 4);
  pl.wd_w = make_div(pl.Ws[0] / 4);
  fwd_divs(pl);
  return WTCONV_OK;
}

// Tile grid and item list of the parameter-gradient pass for tbr-row tiles.
void bw_tiles(const wtconv_desc_t* d, WtBwPlan& pl, int tbr) {
  pl.tbr = tbr;
  pl.tcw = 4;
  pl.item_begin[0] = 0;
  for (int l = 0; l <= d->levels; ++l) {
    pl.tr[l] = ceil_div(pl.Hs[l], tbr);
    pl.tc[l] = ceil_div(pl.Ws[l], 4);
    pl.item_begin[l + 1] = pl.item_begin[l] + (l == 0 ? 1 : 4) * pl.tr[l] * pl.tc[l];
  }
}

// Shared-memory layout of the parameter-gradient pass for `nsets` input sets:
// [input sets][P work areas, or the end-of-channel reduction if larger]
// [mbarriers].  TMA destinations are 128-byte aligned.
void bw_layout(WtBwPlan& pl, int nsets, bool staging) {
  const int P = pl.P, KK = pl.K * pl.K;
  pl.nsets = nsets;
  pl.xr = round_up(P * pl.xbf, 32);
  pl.islot = pl.xr + round_up(P * pl.dbf, 32);
  pl.stage_off = 0;
  int off = nsets * pl.islot;
  if (staging) {  // raw 16-bit x and dy planes of one unit: P * H * W * 2 halves = P * H * W floats
    pl.stage_off = off;
    off += round_up(P * pl.H * pl.W, 32);
  }
  pl.work_off = off;
  long region = (long)P * pl.wf;
  const long red = (long)P * pl.items_per_plane * (KK + 1);  // end-of-channel reduction (reuses the work area)
  if (red > region) region = red;
  pl.red_floats = (int)((region + 3) / 4 * 4);
  pl.mb_off = pl.work_off + pl.red_floats;
  const long smem = 4L * pl.mb_off + 16 + WT_SMEM_SLACK;
  pl.smem_bytes = smem > INT32_MAX ? INT32_MAX : (int)smem;
  pl.tma_bytes = (uint32_t)(4L * P * (pl.xbf + pl.dbf));
}

// Persistent grid and record slots of a gradient plan whose `batches` (units
// per channel) is set; `per_sm` resident CTAs per SM.
wtconv_status_t bw_grid(const wtconv_desc_t* d, WtBwPlan& pl, int per_sm) {
  const long long U = (long long)d->C * pl.batches;
  if (U >= (1 << 24))
    return fail(WTCONV_ERR_UNSUPPORTED, "%lld gradient units exceed the 2^24 index range", U);
  pl.nb_div = make_div(pl.batches > 0 ? pl.batches : 1);
  const long long slots_total = (long long)kNumSms * per_sm;
  pl.grid = (int)(U < slots_total ? U : slots_total);
  if (pl.grid < 1) pl.grid = 1;
  pl.uq = (int)(U / pl.grid);
  pl.ur = (int)(U % pl.grid);
  pl.g_div = make_div(pl.grid);
  pl.nrec = 0;
  for (int i = 0; i < pl.grid && U > 0; ++i) {
    const int ub = bw_unit_begin(pl, i), ue = bw_unit_begin(pl, i + 1);
    const int span = (ue - 1) / pl.batches - ub / pl.batches + 1;
    if (span > pl.nrec) pl.nrec = span;
  }
  return WTCONV_OK;
}

wtconv_status_t plan_bw_compute(const wtconv_desc_t* d, WtBwPlan& pl) {
  memset(&pl, 0, sizeof(pl));
  pl.N = d->N; pl.C = d->C; pl.H = d->H; pl.W = d->W; pl.L = d->levels; pl.K = d->k;
  const int R = d->k / 2, L = d->levels, KK = d->k * d->k;
  level_sizes(d, pl.Hs, pl.Ws);
  // 8x4 tiles (one per thread) when a plane's tiles fit in one CTA and waste
  // no more FMAs than 4x4 tiles would; otherwise 4x4 tiles (two per thread).
  long useful = 0;
  for (int l = 0; l <= L; ++l) useful += (long)(l == 0 ? 1 : 4) * pl.Hs[l] * pl.Ws[l];
  bw_tiles(d, pl, 4);
  const long work4 = 16L * pl.item_begin[L + 1];
  bw_tiles(d, pl, 8);
  const long work8 = 32L * pl.item_begin[L + 1];
  if (pl.item_begin[L + 1] > WT_BW_THREADS || work8 > work4 + useful / 8) bw_tiles(d, pl, 4);
  // Input set: P raw x planes (r zero rows above and below, a 4-float zero
  // margin left and right so rows start 16-byte aligned; the correlation
  // windows read up to r columns beyond the interior) and P raw dy planes (no
  // margin).  The fused level-1/2 analysis reads both up to row/column
  // 4*ceil(H2) - 1, which the tile-rounded extents cover.
  pl.xbf = place(pl.xs[0], 0, pl.tbr * pl.tr[0], pl.tcw * pl.tc[0], R, 4, 1);
  pl.dbf = place(pl.ds[0], 0, pl.tbr * pl.tr[0], pl.tcw * pl.tc[0], 0, 0, 1);
  int off = 0;
  for (int l = 1; l <= L; ++l) {
    if (tiny_band(pl.Hs[l], pl.Ws[l])) {
      off = place_tiny(pl.xs[l], off);
      off = place_tiny(pl.ds[l], off);
      continue;
    }
    // x bands: no left margin (a row's right margin is the next row's left
    // one, 4 zero floats ahead of the buffer serve its first row), so every
    // level's correlation window starts 4 - r floats after a 16-byte boundary
    off = place(pl.xs[l], off + 4, pl.tbr * pl.tr[l], pl.tcw * pl.tc[l] + R, R, 0, 4);
    off = place(pl.ds[l], off, pl.tbr * pl.tr[l], pl.tcw * pl.tc[l], 0, 0, 4);
  }
  pl.wf = round_up(off, 4);
  pl.items_per_plane = pl.item_begin[L + 1];
  pl.nbands = 1 + 4 * L;
  pl.part_stride = pl.nbands * (KK + 1);
  // Tiles per thread.  4-row tiles take one per thread when whole planes
  // fill at least 85 % of the threads and the smaller kernel fits more CTAs
  // per SM (its registers, read from the runtime; at k = 5 80 against 128,
  // three CTAs against two), else two.  On GB300 one per thread was 6-16 %
  // faster on 7 x 7 and 14 x 14 planes, where a CTA fills 94-98 % of its
  // threads, and 20 % slower on 28 x 28 planes at 4-5 levels (54 %).
  pl.mi = 1;
  if (pl.tbr == 4) {
    const int r1 = wt::bw_regs(d->k, 1, d->dtype), r2 = wt::bw_regs(d->k, WT_BW_MAX_ITEMS, d->dtype);
    const long c1 = r1 > 0 ? 65536L / (WT_BW_THREADS * (long)round_up(r1, 8)) : 3;
    const long c2 = r2 > 0 ? 65536L / (WT_BW_THREADS * (long)round_up(r2, 8)) : 2;
    const bool fills = pl.items_per_plane <= WT_BW_THREADS &&
                       (WT_BW_THREADS / pl.items_per_plane) * pl.items_per_plane * 100 >= 85 * WT_BW_THREADS;
    if (!fills || c1 <= c2) pl.mi = WT_BW_MAX_ITEMS;
  }
  const int slots = pl.mi * WT_BW_THREADS;
  if (pl.items_per_plane > slots)
    return fail(WTCONV_ERR_UNSUPPORTED, "plane %dx%d has %d gradient tiles (max %d per CTA)", d->H, d->W,
                pl.items_per_plane, slots);
  const long plane_bytes = 4L * (2 * (pl.xbf + pl.dbf) + pl.wf) + 256;
  int P = slots / pl.items_per_plane;
  const int fit = (int)(kBwBudget / plane_bytes);
  if (P > fit) P = fit < 1 ? 1 : fit;
  if (d->N > 0 && P > d->N) P = d->N;
  if (P < 1) P = 1;
  pl.P = P;
  // 16-bit planes that are whole 8-byte chunks get a staging area for their
  // raw planes (used when the tensors are aligned enough; see set_bulk).
  const bool staging = d->dtype != WTCONV_F32 && (2L * d->H * d->W) % 8 == 0;
  bw_layout(pl, 2, false);
  if (pl.smem_bytes > kMaxSmemPerBlock) {
    bw_layout(pl, 1, false);
    if (pl.smem_bytes > kMaxSmemPerBlock)
      return fail(WTCONV_ERR_UNSUPPORTED, "plane %dx%d with %d levels needs %d B of shared memory (max %d)",
                  d->H, d->W, L, pl.smem_bytes, kMaxSmemPerBlock);
  }
  for (int l = 0; l <= L; ++l) {
    pl.an_pp[l] = make_div(pl.Hs[l] * pl.Ws[l]);
    pl.an_w[l] = make_div(pl.Ws[l]);
    pl.tiles[l] = make_div(pl.tr[l] * pl.tc[l]);
    pl.tcd[l] = make_div(pl.tc[l]);
  }
  if (L >= 2) {  // the fused level-1/2 pass walks the level-2 grid
    pl.an_pp[2] = make_div(pl.Hs[2] * pl.Ws[2]);
    pl.an_w[2] = make_div(pl.Ws[2]);
  }
  pl.ipp = make_div(pl.items_per_plane);
  // Resident CTAs per SM from the occupancy calculator (registers and shared
  // memory); without a device, from shared memory alone, at most 2.  Two
  // input sets let float32 units stream in while the previous one is
  // processed (one set when two do not fit).
  auto per_sm_of = [&](const WtBwPlan& q) {
    int n = wt::bw_ctas_per_sm(q, d->dtype);
    if (n <= 0) {
      n = (int)(kSmemPerSm / (q.smem_bytes + 1024));
      if (n > 2) n = 2;
    }
    return n < 1 ? 1 : n;
  };
  // 16-bit activations are loaded synchronously, so they need one input set.
  if (d->dtype != WTCONV_F32) {
    bw_layout(pl, 1, staging);
    if (pl.smem_bytes > kMaxSmemPerBlock) bw_layout(pl, 1, false);
  }
  int per_sm = per_sm_of(pl);
  // float32: one input set instead of two where that fits more CTAs per SM
  // (the next unit's boxes then follow the unit, prefetched into L2 first).
  if (d->dtype == WTCONV_F32 && pl.nsets == 2) {
    WtBwPlan one = pl;
    bw_layout(one, 1, false);
    const int per_sm1 = per_sm_of(one);
    if (per_sm1 > per_sm) {
      pl = one;
      per_sm = per_sm1;
    }
  }
  // Persistent grid: every resident CTA slot, at most one CTA per unit.
  pl.batches = d->N > 0 ? ceil_div(d->N, P) : 0;
  return bw_grid(d, pl, per_sm);
}

// Plan of the fused backward (input gradient and parameter gradients in one
// kernel, planes that fit one CTA): the parameter-gradient plan's tiles,
// items and units, with the dy buffers widened for the input-gradient
// phases (an r-row, 4-column zero margin around the dy plane and every dy
// band, so the band convolutions and the base convolution read their halo
// from it), plus the input gradient's Z buffers and rotated folded weights.
// Shared memory: [input sets: P x planes, P dy planes][work area: P x (x
// pyramid, dy pyramid, Z buffers), or the end-of-channel reduction][weights]
// [mbarriers].  Two input sets and two CTAs per SM are preferred, then one
// set, then fewer planes per unit; layers that cannot keep two CTAs per SM
// are refused (the caller then runs the two separate passes).
wtconv_status_t plan_bwf_compute(const wtconv_desc_t* d, WtBwPlan& pl, WtFwdPlan& fp) {
  const wtconv_status_t st = plan_bw(d, pl);  // fails for planes beyond one CTA
  if (st != WTCONV_OK) return st;
  // 4-row correlation tiles (deep pyramids, small planes): the fused kernel
  // measured no faster than the two passes there, and is not built for them.
  if (pl.tbr != 8)
    return fail(WTCONV_ERR_UNSUPPORTED, "plane %dx%d takes 4-row gradient tiles: no fused backward kernel",
                d->H, d->W);
  const int R = d->k / 2, L = d->levels, KK = d->k * d->k;
  memset(&fp, 0, sizeof(fp));
  fp.N = d->N; fp.C = d->C; fp.H = d->H; fp.W = d->W; fp.L = L; fp.K = d->k;
  for (int l = 0; l <= L; ++l) {
    fp.Hs[l] = pl.Hs[l];
    fp.Ws[l] = pl.Ws[l];
  }
  // Half-height final tiles: with 256 threads and planes of at most 64 x 64,
  // they never take more rounds than full-height ones and each is cheaper.
  const int tp = WT_TP / 2;
  fp.ftp = tp;
  fp.ftr = ceil_div(pl.Hs[1], tp);
  fp.ftc = ceil_div(pl.Ws[1], WT_TQ);
  const int rows0 = std::max(pl.tbr * pl.tr[0], 2 * tp * fp.ftr);
  const int cols0 = std::max(4 * pl.tc[0], 2 * WT_TQ * fp.ftc);
  pl.xbf = place(pl.xs[0], 0, pl.tbr * pl.tr[0], 4 * pl.tc[0], R, 4, 1);
  pl.dbf = place(pl.ds[0], 0, rows0, cols0, R, 4, 1, cols0 + 8);
  // Work area: per level the x bands, the dy bands and (after all levels)
  // the Z buffers.  With pad, the dy bands' strides are 4 mod 8 floats, so
  // the 4-row band-convolution tiles of a warp start 16 banks apart; the
  // padding is kept only where it costs no planes per unit.
  auto work_geometry = [&](bool pad) {
    int off = 0;
    fp.zbegin[1] = 0;
    for (int l = 1; l <= L; ++l) {
      fp.ztr[l] = ceil_div(pl.Hs[l], WT_ZT);
      fp.ztc[l] = ceil_div(pl.Ws[l], WT_ZT);
      // x bands: no left margin.  A row's right margin (at least r zero
      // columns) is the next row's left one, and 4 zero floats ahead of the
      // buffer serve its first row; the correlation then reads every level
      // at the same offset from a 16-byte boundary.
      off = place(pl.xs[l], off + 4, pl.tbr * pl.tr[l], 4 * pl.tc[l] + R, R, 0, 4);
      const int dcols = std::max(4 * pl.tc[l], WT_ZT * fp.ztc[l]);
      off = place(pl.ds[l], off, std::max(pl.tbr * pl.tr[l], WT_ZT * fp.ztr[l]), dcols, R, 4, 4,
                  pad ? pad48(dcols + 8) : 0);
      fp.zbegin[l + 1] = fp.zbegin[l] + 4 * fp.ztr[l] * fp.ztc[l];
    }
    fp.zipp = fp.zbegin[L + 1];
    for (int l = 1; l <= L; ++l) {
      // Z^l: written at p < H_l, q < W_l; read by the final tiles at
      // (p >> (l-1), q >> (l-1)) for every level-1 position of the tile grid.
      const int fr = ((tp * fp.ftr - 1) >> (l - 1)) + 1, fc = ((WT_TQ * fp.ftc - 1) >> (l - 1)) + 1;
      off = place(fp.zb[l], off, std::max(pl.Hs[l], fr), std::max(pl.Ws[l], fc), 0, 0, 4);
    }
    pl.wf = fp.wf = round_up(off, 4);
  };
  fp.xf = pl.dbf;
  fp.w_band = round_up(KK, 4);
  const int wfloats = (1 + 4 * L) * fp.w_band;
  // 16-bit planes that are whole 8-byte chunks get a staging area for their
  // raw planes, and one input set (used when the tensors are aligned enough);
  // where the staging area would cost the second CTA per SM, the planes are
  // loaded element-wise instead, without one.
  bool staging = d->dtype != WTCONV_F32 && (2L * d->H * d->W) % 8 == 0;
  auto layout = [&](int P, int nsets) {
    pl.P = P;
    pl.nsets = nsets;
    pl.xr = round_up(P * pl.xbf, 32);
    pl.islot = pl.xr + round_up(P * pl.dbf, 32);
    pl.stage_off = nsets * pl.islot;
    pl.work_off = pl.stage_off + (staging ? round_up(P * d->H * d->W, 32) : 0);
    long region = (long)P * pl.wf;
    const long red = (long)P * pl.items_per_plane * (KK + 1);
    if (red > region) region = red;
    pl.red_floats = (int)((region + 3) / 4 * 4);
    fp.w_off = pl.work_off + pl.red_floats;
    pl.mb_off = round_up(fp.w_off + wfloats, 2);
    const long smem = 4L * pl.mb_off + 16 + WT_SMEM_SLACK;
    pl.smem_bytes = smem > INT32_MAX ? INT32_MAX : (int)smem;
    pl.tma_bytes = (uint32_t)(4L * P * (pl.xbf + pl.dbf));
  };
  const long two_per_sm = kSmemPerSm / 2 - 1024 - kStaticSmem;
  const int p_max = pl.P;
  auto fit = [&]() {
    for (int q = p_max; q >= 1; --q)
      for (int ns = staging ? 1 : 2; ns >= 1; --ns) {
        layout(q, ns);
        if (pl.smem_bytes <= two_per_sm) return true;
      }
    return false;
  };
  work_geometry(false);
  bool found = fit();
  if (!found && staging) {
    staging = false;
    found = fit();
  }
  const int P0 = pl.P, ns0 = pl.nsets;
  if (found) {
    work_geometry(true);
    if (!fit() || pl.P != P0 || pl.nsets != ns0) {
      work_geometry(false);
      layout(P0, ns0);
    }
  }
  // One 256-thread CTA per SM leaves too few warps to hide the phases'
  // latency: such layers run the two separate passes (which keep 2-3 CTAs
  // per SM) instead.
  if (!found)
    return fail(WTCONV_ERR_UNSUPPORTED, "plane %dx%d with %d levels: the fused backward's working set leaves "
                "one CTA per SM", d->H, d->W, L);
  for (int l = 0; l <= L; ++l) fp.lev[l] = pl.ds[l];
  fp.P = pl.P;
  fwd_divs(fp);
  pl.batches = d->N > 0 ? ceil_div(d->N, pl.P) : 0;
  int per_sm = wt::bwf_ctas_per_sm(pl, fp, d->dtype);
  if (per_sm == 1)
    return fail(WTCONV_ERR_UNSUPPORTED, "k=%d: the fused backward's registers leave one CTA per SM", d->k);
  if (per_sm <= 0) {
    per_sm = (int)(kSmemPerSm / (pl.smem_bytes + 1024));
    if (per_sm > 2) per_sm = 2;
  }
  return bw_grid(d, pl, per_sm < 1 ? 1 : per_sm);
}

// Windowed parameter-gradient geometry for th x tw tiles and tbr-row
// correlation tiles; pl.halo set.  x window: (th + 2h) x (tw + 2h) pixels
// with r zero rows above and below and a 4-float margin left and right (the
// float32 box copy fills exactly this); dy tile: th x tw, no margin.  x
// level buffers: no top margin, a column margin (-zo) mod 4 that puts every
// correlation window's first column 4 - r floats after a 16-byte boundary
// (as in the raw window, whose tile origin is zo[0] = h), and room for the
// rows and columns the last correlation tiles read past the window; dy level
// buffers: the tile's coefficients rounded up to whole correlation tiles
// (the rounding margin stays zero).  Both strides of the bands are 4 mod 8
// floats: the 4-row correlation tiles of a warp then start 16 banks apart
// from one tile row to the next instead of on the same banks.
void bw_win_geometry(const wtconv_desc_t* d, WtBwPlan& pl, int th, int tw, int tbr) {
  const int R = d->k / 2, L = d->levels, h = pl.halo;
  pl.th = th;
  pl.tw = tw;
  pl.tbr = tbr;
  pl.tcw = 4;
  pl.Hs[0] = th + 2 * h;
  pl.Ws[0] = tw + 2 * h;
  for (int l = 0; l <= L; ++l) {
    pl.Hs[l] = pl.Hs[0] >> l;
    pl.Ws[l] = pl.Ws[0] >> l;
    pl.dHs[l] = th >> l;
    pl.dWs[l] = tw >> l;
  }
  pl.item_begin[0] = 0;
  for (int l = 0; l <= L; ++l) {
    pl.tr[l] = ceil_div(th >> l, tbr);
    pl.tc[l] = ceil_div(tw >> l, 4);
    pl.item_begin[l + 1] = pl.item_begin[l] + (l == 0 ? 1 : 4) * pl.tr[l] * pl.tc[l];
  }
  pl.items_per_plane = pl.item_begin[L + 1];
  pl.xbf = place(pl.xs[0], 0, pl.Hs[0], pl.Ws[0], R, 4, 1);
  pl.dbf = place(pl.ds[0], 0, th, tw, 0, 0, 1);
  pl.zo[0] = h;
  int off = 0;
  for (int l = 1; l <= L; ++l) {
    const int zo = h >> l;
    pl.zo[l] = zo;
    WtBuf& b = pl.xs[l];
    b.off = off;
    b.prow = 0;
    b.pcol = (4 - zo % 4) % 4;
    const int rows = std::max(pl.Hs[l], zo + tbr * pl.tr[l] + R);
    const int cols = std::max(b.pcol + pl.Ws[l], zo + 4 * pl.tc[l] + R + b.pcol);
    b.stride = pad48(cols);
    b.band = rows * b.stride;
    off += 4 * b.band;
    off = place(pl.ds[l], off, tbr * pl.tr[l], 4 * pl.tc[l], 0, 0, 4, pad48(4 * pl.tc[l]));
  }
  pl.wf = round_up(off, 4);
}

// Shared-memory layout of a windowed gradient plan: [input sets: P x windows,
// then P dy tiles][16-bit staging: raw x windows, then raw dy tiles][work
// area: P pyramid pairs, or the end-of-channel reduction if larger][mbarriers].
void bw_win_layout(WtBwPlan& pl, int P, int nsets, int load) {
  const int KK = pl.K * pl.K;
  pl.P = P;
  pl.nsets = nsets;
  pl.xr = round_up(P * pl.xbf, 32);
  pl.islot = pl.xr + round_up(P * pl.dbf, 32);
  int off = nsets * pl.islot;
  pl.stage_off = off;
  pl.stage_dx = 0;
  if (load == 2) {
    pl.stage_dx = round_up((P * pl.Hs[0] * pl.Ws[0] + 1) / 2, 32);
    off += pl.stage_dx + round_up((P * pl.th * pl.tw + 1) / 2, 32);
  }
  pl.work_off = off;
  long region = (long)P * pl.wf;
  const long red = (long)P * pl.items_per_plane * (KK + 1);
  if (red > region) region = red;
  pl.red_floats = (int)((region + 3) / 4 * 4);
  pl.mb_off = pl.work_off + pl.red_floats;
  const long smem = 4L * pl.mb_off + 16 + WT_SMEM_SLACK;
  pl.smem_bytes = smem > INT32_MAX ? INT32_MAX : (int)smem;
  pl.tma_bytes = load == 1 ? (uint32_t)(4L * P * (pl.xbf + pl.dbf))
                           : load == 2 ? (uint32_t)(2L * P * (pl.Hs[0] * pl.Ws[0] + pl.th * pl.tw)) : 0u;
}

// Windowed parameter-gradient plan for planes too large for plan_bw.
// `load` as for plan_win.  Tile, correlation-tile height, planes per unit and
// input sets minimise the modelled time of the call, as in plan_win: phase
// rounds of the 256 threads (both pyramids, then one or two correlation
// items per thread) times the number of units, weighted by the CTAs that fit
// an SM by shared memory and by the kernel's registers.  The weights (4-row
// correlation items at 0.6 of their FMA count, 1 / 2 / 3 CTAs per SM at
// 1.6 / 1.0 / 0.8, one float32 input set at 0.9 of two) were fitted to a
// sweep of forced tilings on a GB300 (224 x 224 planes at levels 1-4 and
// k = 5, 7; 128, 384 and 512-pixel planes; float32 and float16), where the
// model's choice came within 0.3 % of the fastest measured tiling on seven
// of eight shapes and within 6.3 % on the eighth.
wtconv_status_t plan_bw_win_compute(const wtconv_desc_t* d, WtBwPlan& pl, int load) {
  memset(&pl, 0, sizeof(pl));
  pl.N = d->N; pl.C = d->C; pl.H = d->H; pl.W = d->W; pl.L = d->levels; pl.K = d->k;
  const int R = d->k / 2, L = d->levels, KK = d->k * d->k, S = 1 << L;
  pl.win = 1;
  pl.win_load = load;
  pl.halo = round_up(R * S, 8);
  const int h = pl.halo, A = S > 8 ? S : 8;
  const int thmax = round_up(d->H, A), twmax = round_up(d->W, A);
  const int NT = WT_BW_THREADS;
  const long c12 = 100, c3 = 30, cunit = 600 + 200L * (L > 2 ? L - 2 : 0);
  const int Pmax = d->N < 1 ? 1 : (d->N < 8 ? d->N : 8);
  double best = -1.0;
  int bth = 0, btw = 0, btr = 0, bP = 0, bns = 0;
  for (int T = A;; T += A) {
    const int th = T < thmax ? T : thmax, tw = T < twmax ? T : twmax;
    if (tw + 2 * h + 8 > 256 || th + 2 * h + 2 * R > 256) break;  // one box per window and plane
    for (int tbr = 8; tbr >= 4; tbr /= 2) {
      bw_win_geometry(d, pl, th, tw, tbr);
      const int slots = (tbr == 8 ? 1 : WT_BW_MAX_ITEMS) * NT;
      const int n12x = L >= 2 ? pl.Hs[2] * pl.Ws[2] : pl.Hs[1] * pl.Ws[1];
      const int n12d = L >= 2 ? pl.dHs[2] * pl.dWs[2] : pl.dHs[1] * pl.dWs[1];
      const long citem = (tbr == 8 ? 4L * tbr * KK : 12L * tbr * KK / 5) + 200;
      const int regs = wt::bw_win_regs(d->k, tbr, d->dtype);
      const long ctas_r = regs > 0 ? 65536L / (NT * (long)round_up(regs, 8)) : 3;
      for (int q = 1; q <= Pmax && q * pl.items_per_plane <= slots; ++q) {
        for (int ns = (load == 1 ? 2 : 1); ns >= 1; --ns) {
          bw_win_layout(pl, q, ns, load);
          if (pl.smem_bytes > kMaxSmemPerBlock) continue;
          long ctas = kSmemPerSm / (pl.smem_bytes + 1024);
          if (ctas > ctas_r) ctas = ctas_r;
          if (ctas > 3) ctas = 3;
          long cost = ceil_div(q * n12x, NT) * c12 + ceil_div(q * n12d, NT) * c12 +
                      ceil_div(q * pl.items_per_plane, NT) * citem + cunit;
          for (int l = 3; l <= L; ++l)
            cost += (ceil_div(q * pl.Hs[l] * pl.Ws[l], NT) + ceil_div(q * pl.dHs[l] * pl.dWs[l], NT)) * c3;
          if (load == 0) cost += ceil_div(q * (pl.Hs[0] * pl.Ws[0] + th * tw) / 4, NT) * 60;
          const double units = (double)ceil_div(d->N > 0 ? d->N : 1, q) * ceil_div(d->H, th) * ceil_div(d->W, tw);
          const double occ = ctas >= 3 ? 0.8 : ctas == 2 ? 1.0 : 1.6;
          const double one_set = (load == 1 && ns == 1) ? 0.9 : 1.0;
          const double total = (double)cost * units * occ * one_set;
          if (best < 0 || total < best * (1 - 1e-9)) {
            best = total;
            bth = th; btw = tw; btr = tbr; bP = q; bns = ns;
          }
        }
      }
    }
    if (th == thmax && tw == twmax) break;
  }
  if (best < 0)
    return fail(WTCONV_ERR_UNSUPPORTED,
                "plane %dx%d does not fit one CTA for the parameter gradient, and neither does the smallest "
                "%dx%d tile with its %d-pixel halo (levels %d, k %d)", d->H, d->W, A, A, h, L, d->k);
  bw_win_geometry(d, pl, bth, btw, btr);
  bw_win_layout(pl, bP, bns, load);
  pl.groups = d->N > 0 ? ceil_div(d->N, bP) : 0;
  pl.nty = ceil_div(d->H, bth);
  pl.ntx = ceil_div(d->W, btw);
  if ((long long)pl.groups * pl.nty * pl.ntx >= (1 << 24))
    return fail(WTCONV_ERR_UNSUPPORTED, "too many gradient tiles per channel");
  pl.batches = pl.groups * pl.nty * pl.ntx;
  pl.nbands = 1 + 4 * L;
  pl.part_stride = pl.nbands * (KK + 1);
  for (int l = 0; l <= L; ++l) {
    pl.an_pp[l] = make_div(pl.Hs[l] * pl.Ws[l]);
    pl.an_w[l] = make_div(pl.Ws[l]);
    pl.dn_pp[l] = make_div(pl.dHs[l] * pl.dWs[l]);
    pl.dn_w[l] = make_div(pl.dWs[l]);
    pl.tiles[l] = make_div(pl.tr[l] * pl.tc[l]);
    pl.tcd[l] = make_div(pl.tc[l]);
  }
  pl.ipp = make_div(pl.items_per_plane);
  pl.wd_vec = 4;
  pl.wd_pp = make_div(pl.Hs[0] * pl.Ws[0] / 4);
  pl.wd_w = make_div(pl.Ws[0] / 4);
  pl.dwd_pp = make_div(pl.th * pl.tw / 4);
  pl.dwd_w = make_div(pl.tw / 4);
  int per_sm = wt::bw_win_ctas_per_sm(pl, d->dtype);
  if (per_sm <= 0) {
    per_sm = (int)(kSmemPerSm / (pl.smem_bytes + 1024));
    if (per_sm > 2) per_sm = 2;
  }
  return bw_grid(d, pl, per_sm < 1 ? 1 : per_sm);
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the
// library does not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tensor map over a float32 NCHW tensor, dimensions (W, H, C, N) innermost
// first, with box (box_w, box_h, 1, P): one box is P planes of one channel
// with a margin, landing in shared memory as P consecutive padded planes.
// Out-of-range elements read as zero.  Returns false if TMA cannot be used.
bool encode_plane_map(CUtensorMap* m, const void* base, const wtconv_desc_t* d, int box_w, int box_h, int P) {
  if (d->dtype != WTCONV_F32 || (d->W % 4) != 0 || !aligned(base, 16)) return false;
  if (box_w > 256 || box_h > 256 || P > 256 || (box_w % 4) != 0) return false;
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d->W, (cuuint64_t)d->H, (cuuint64_t)d->C, (cuuint64_t)d->N};
  const cuuint64_t strides[3] = {4ull * d->W, 4ull * d->W * d->H, 4ull * d->W * d->H * d->C};
  const cuuint32_t box[4] = {(cuuint32_t)box_w, (cuuint32_t)box_h, 1u, (cuuint32_t)P};
  const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over a 16-bit NCHW tensor for the windowed pass: box
// (box_w, box_h, 1, P) elements, landing as P consecutive raw windows.
// Rows must be whole 16-byte chunks (W % 8 == 0) and box_w a multiple of 8.
bool encode_map16(CUtensorMap* m, const void* base, const wtconv_desc_t* d, int box_w, int box_h, int P) {
  if (d->dtype == WTCONV_F32 || (d->W % 8) != 0 || !aligned(base, 16)) return false;
  if (box_w > 256 || box_h > 256 || P > 256 || (box_w % 8) != 0) return false;
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)d->W, (cuuint64_t)d->H, (cuuint64_t)d->C, (cuuint64_t)d->N};
  const cuuint64_t strides[3] = {2ull * d->W, 2ull * d->W * d->H, 2ull * d->W * d->H * d->C};
  const cuuint32_t box[4] = {(cuuint32_t)box_w, (cuuint32_t)box_h, 1u, (cuuint32_t)P};
  const cuuint32_t es[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapDataType t =
      d->dtype == WTCONV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return fn(m, t, 4, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Window load mode for source `src`: box copies when its rows are whole
// 16-byte chunks and it is 16-byte aligned, else plain loads.
int win_load_mode(const wtconv_desc_t* d, const void* src) {
  if (!aligned(src, 16)) return 0;
  if (d->dtype == WTCONV_F32) return d->W % 4 == 0 ? 1 : 0;
  return d->W % 8 == 0 ? 2 : 0;
}

// Plan of the parameter-gradient pass: whole planes when both pyramids fit
// one CTA, else tiles with a halo on x.  Box copies need x and dy 16-byte
// aligned with 16-byte rows.
wtconv_status_t plan_bw_any(const wtconv_desc_t* d, WtBwPlan& pl, const void* x, const void* dy) {
  const wtconv_status_t st = plan_bw(d, pl);
  if (st != WTCONV_ERR_UNSUPPORTED) return st;
  const int mx = win_load_mode(d, x), md = win_load_mode(d, dy);
  return plan_bw_win(d, pl, mx == md ? mx : 0);
}

// Plan of the forward / input-gradient pass: whole planes when a plane and
// its pyramid fit one CTA, else output tiles with a halo.
wtconv_status_t plan_any(const wtconv_desc_t* d, WtFwdPlan& pl, const void* src) {
  const wtconv_status_t st = plan_fwd(d, pl);
  if (st != WTCONV_ERR_UNSUPPORTED) return st;
  return plan_win(d, pl, win_load_mode(d, src));
}

wtconv_status_t check_act(const void* p, const char* name, const wtconv_desc_t* d) {
  if (!p) return fail(WTCONV_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, elem_size(d->dtype)))
    return fail(WTCONV_ERR_MISALIGNED, "%s is not aligned to its element size", name);
  return WTCONV_OK;
}

wtconv_status_t check_param(const void* p, const char* name, bool nullable) {
  if (!p) return nullable ? WTCONV_OK : fail(WTCONV_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, 4)) return fail(WTCONV_ERR_MISALIGNED, "%s is not 4-byte aligned", name);
  return WTCONV_OK;
}

int vec_ok(const wtconv_desc_t* d, const void* a, const void* b) {
  const int v = (int)(16 / elem_size(d->dtype));
  return (d->W % v == 0) && aligned(a, 16) && (b == nullptr || aligned(b, 16));
}

// Plane-load loop divisors: 16-byte items when the rows allow it, else elements.
template <typename Plan>
void set_load_divs(Plan& pl, const wtconv_desc_t* d, int vec) {
  pl.vec_ok = vec;
  const int per_row = vec ? d->W / (int)(16 / elem_size(d->dtype)) : d->W;
  pl.ld_pp = make_div(d->H * per_row);
  pl.ld_w = make_div(per_row);
}

// 16-bit planes are staged raw and widened in shared memory: by one bulk copy
// per plane when a plane is a whole number of 16-byte chunks and the tensor is
// 16-byte aligned (mode 1), else by 8-byte cp.async chunks when a plane is a
// whole number of 8-byte chunks and the tensor is 8-byte aligned (mode 2).
template <typename Plan>
void set_bulk(Plan& pl, const wtconv_desc_t* d, const void* src, long capacity_bytes) {
  const long plane = 2L * d->H * d->W;
  pl.use_bulk = 0;
  if (d->dtype != WTCONV_F32 && plane * pl.P <= capacity_bytes) {
    if (plane % 16 == 0 && aligned(src, 16) && plane * pl.P < (1L << 20)) pl.use_bulk = 1;
    else if (plane % 8 == 0 && aligned(src, 8)) pl.use_bulk = 2;
  }
  pl.bulk_bytes = (uint32_t)plane;
  pl.cp_pp = make_div((int)(plane / 8 > 0 ? plane / 8 : 1));
  pl.wd_vec = d->W % 4 == 0 ? 4 : (d->W % 2 == 0 ? 2 : 1);
  const int per_row = d->W / pl.wd_vec;
  pl.wd_pp = make_div(d->H * per_row);
  pl.wd_w = make_div(per_row);
}

size_t bw_workspace_bytes(const WtBwPlan& pl) {
  const size_t bytes = (size_t)pl.grid * pl.nrec * pl.part_stride * sizeof(float);
  return (bytes + 255) / 256 * 256;
}

#define WT_TRY(expr)                  \
  do {                                \
    wtconv_status_t st_ = (expr);     \
    if (st_ != WTCONV_OK) return st_; \
  } while (0)

// Pointer-dependent parts of a windowed plan: the box tensor map (re-planned
// for plain loads if it cannot be encoded) and the plain-load divisors.
wtconv_status_t prepare_win(const wtconv_desc_t* d, WtFwdPlan& pl, CUtensorMap* m, const void* src,
                            const void* dst) {
  bool boxed = true;
  if (pl.win_load == 1)
    boxed = encode_plane_map(m, src, d, pl.lev[0].stride, pl.lev[0].band / pl.lev[0].stride, pl.P);
  else if (pl.win_load == 2)
    boxed = encode_map16(m, src, d, pl.Ws[0], pl.Hs[0], pl.P);
  if (!boxed) WT_TRY(plan_win(d, pl, 0));
  pl.vec_ok = vec_ok(d, src, dst);
  const int per_row = pl.vec_ok ? pl.Ws[0] / (int)(16 / elem_size(d->dtype)) : pl.Ws[0];
  pl.ld_pp = make_div(pl.Hs[0] * per_row);
  pl.ld_w = make_div(per_row);
  return WTCONV_OK;
}

// ---- Coarse-level split ------------------------------------------------------
// A layer whose tile window does not fit one CTA runs as two layers (the
// reasoning and the element-wise kernels are in wtconv_split.cu): the fine
// pass, levels 1..s and the base convolution on the full planes; and the
// coarse layer, levels s+1..L and no base convolution, on the float32 level-s
// low-pass planes, whose output is added back block-replicated.  The coarse
// layer's level l' is the original level s + l': same kernels w_sub, and
// wavelet scales times 4^-s, so that its folded weights 4^-l' * s' * W equal
// the original 4^-(s+l') * s * W; its wavelet-scale gradient is therefore 4^s
// times the original's.

int box_mode(const wtconv_desc_t* d) {
  if (d->dtype == WTCONV_F32) return d->W % 4 == 0 ? 1 : 0;
  return d->W % 8 == 0 ? 2 : 0;
}

// Whether a forward / input-gradient pass has a plan whatever the pointers'
// alignment (whole planes, or tiles under every load mode).
bool fwd_plannable(const wtconv_desc_t* d) {
  WtFwdPlan pl;
  if (plan_fwd(d, pl) == WTCONV_OK) return true;
  const int m = box_mode(d);
  return plan_win(d, pl, 0) == WTCONV_OK && (m == 0 || plan_win(d, pl, m) == WTCONV_OK);
}

bool bw_plannable(const wtconv_desc_t* d) {
  WtBwPlan pl;
  if (plan_bw(d, pl) == WTCONV_OK) return true;
  const int m = box_mode(d);
  return plan_bw_win(d, pl, 0) == WTCONV_OK && (m == 0 || plan_bw_win(d, pl, m) == WTCONV_OK);
}

wtconv_desc_t fine_desc(const wtconv_desc_t* d, int s) {
  wtconv_desc_t f = *d;
  f.levels = s;
  return f;
}

// The coarse layer: float32 planes of ceil(H / 2^s) x ceil(W / 2^s).
wtconv_desc_t coarse_desc(const wtconv_desc_t* d, int s) {
  wtconv_desc_t c = *d;
  c.H = (int)(((long)d->H + (1L << s) - 1) >> s);
  c.W = (int)(((long)d->W + (1L << s) - 1) >> s);
  c.levels = d->levels - s;
  c.dtype = WTCONV_F32;
  return c;
}

// Levels of the fine pass for a layer that has no plan of its own: the
// largest s whose fine pass has a plan and whose coarse layer has one or
// splits in turn (0 if the layer needs no split, or none works).  Each split
// lowers the level count, so the recursion ends.
int split_levels(const wtconv_desc_t* d, bool grad) {
  bool (*plannable)(const wtconv_desc_t*) = grad ? bw_plannable : fwd_plannable;
  if (plannable(d)) return 0;
  for (int s = d->levels - 1; s >= 1; --s) {
    const wtconv_desc_t f = fine_desc(d, s), c = coarse_desc(d, s);
    if (plannable(&f) && (plannable(&c) || split_levels(&c, grad) > 0)) return s;
  }
  return 0;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace of a split call, byte offsets (each 256-byte aligned):
//   fine   the fine pass's own workspace (parameter gradients only);
//   ll     low-pass planes of x (forward) or dy (input gradient) or x (parameter gradients);
//   ll2    low-pass planes of dy (parameter gradients);
//   carry  the coarse layer's output (forward, input gradient);
//   zeros  the coarse layer's base kernels and base scales (C*k*k + C zeros);
//   sw     its wavelet scales ((L-s)*4C);
//   dummy  its base-kernel and base-scale gradients, discarded (parameter gradients);
//   sub    its own workspace.
struct SplitLayout {
  size_t fine = 0, fine_bytes = 0, ll = 0, ll2 = 0, carry = 0, zeros = 0, sw = 0, dummy = 0, sub = 0, total = 0;
};

SplitLayout split_layout(const wtconv_desc_t* d, int op, int s) {
  SplitLayout w;
  const wtconv_desc_t f = fine_desc(d, s), c = coarse_desc(d, s);
  const bool grad = op == WTCONV_OP_BWD_WEIGHT;
  const size_t KK = (size_t)d->k * d->k, C = (size_t)d->C;
  const size_t ll_bytes = 4 * (size_t)d->N * C * (size_t)c.H * (size_t)c.W;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  if (grad) {
    w.fine_bytes = align256(wtconv_workspace_size(&f, WTCONV_OP_BWD_WEIGHT));
    w.fine = take(w.fine_bytes);
  }
  w.ll = take(ll_bytes);
  if (grad) w.ll2 = take(ll_bytes);
  else w.carry = take(ll_bytes);
  w.zeros = take(4 * (C * KK + C));
  w.sw = take(4 * (size_t)(d->levels - s) * 4 * C);
  if (grad) w.dummy = take(4 * (C * KK + C));
  w.sub = take(wtconv_workspace_size(&c, grad ? WTCONV_OP_BWD_WEIGHT : op));
  w.total = off;
  return w;
}

size_t split_bytes(const wtconv_desc_t* d, int op) {
  const int s = split_levels(d, op == WTCONV_OP_BWD_WEIGHT);
  return s > 0 ? split_layout(d, op, s).total : 0;
}

wtconv_status_t split_workspace_ok(const SplitLayout& w, void* ws, size_t ws_bytes) {
  if (!ws || ws_bytes < w.total)
    return fail(WTCONV_ERR_WORKSPACE, "workspace of %zu B given, %zu B needed (coarse-level split)",
                ws ? ws_bytes : 0, w.total);
  if (!aligned(ws, 256)) return fail(WTCONV_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  return WTCONV_OK;
}

// Zero base kernels and scales, and the scaled wavelet scales, of the coarse layer.
wtconv_status_t split_params(const wtconv_desc_t* d, int s, const float* wavelet_scale, char* ws,
                             const SplitLayout& w, cudaStream_t st) {
  const size_t KK = (size_t)d->k * d->k, C = (size_t)d->C;
  cudaError_t e = cudaMemsetAsync(ws + w.zeros, 0, 4 * (C * KK + C), st);
  if (e == cudaSuccess)
    e = wt::launch_scale(wavelet_scale + (size_t)s * 4 * C, reinterpret_cast<float*>(ws + w.sw),
                         (d->levels - s) * 4 * d->C, ldexpf(1.f, -2 * s), st);
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "coarse-level split: %s", cudaGetErrorString(e));
  return WTCONV_OK;
}

// Forward (grad = false) or input gradient (grad = true) of a split layer.
wtconv_status_t split_fwd(const wtconv_desc_t* d, int s, bool grad, const void* x, const float* w_base,
                          const float* b_base, const float* w_sub, const float* base_scale,
                          const float* wavelet_scale, void* y, void* ws, size_t ws_bytes, cudaStream_t st) {
  const SplitLayout w = split_layout(d, grad ? WTCONV_OP_BWD_DATA : WTCONV_OP_FWD, s);
  WT_TRY(split_workspace_ok(w, ws, ws_bytes));
  const wtconv_desc_t f = fine_desc(d, s), c = coarse_desc(d, s);
  char* b = static_cast<char*>(ws);
  float* ll = reinterpret_cast<float*>(b + w.ll);
  float* carry = reinterpret_cast<float*>(b + w.carry);
  const float* wb0 = reinterpret_cast<const float*>(b + w.zeros);
  const float* sb0 = wb0 + (size_t)d->C * d->k * d->k;
  const float* sw = reinterpret_cast<const float*>(b + w.sw);
  const float* wsub_c = w_sub + (size_t)s * 4 * d->C * d->k * d->k;
  if (grad) {
    WT_TRY(wtconv_bwd_data(&f, x, w_base, w_sub, base_scale, wavelet_scale, y, nullptr, 0, st));
  } else {
    WT_TRY(wtconv_fwd(&f, x, w_base, b_base, w_sub, base_scale, wavelet_scale, y, nullptr, 0, st));
  }
  WT_TRY(split_params(d, s, wavelet_scale, b, w, st));
  cudaError_t e = wt::launch_lowpass(d->dtype, x, ll, (long long)d->N * d->C, d->H, d->W, s, st);
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "coarse-level split: %s", cudaGetErrorString(e));
  if (grad) {
    WT_TRY(wtconv_bwd_data(&c, ll, wb0, wsub_c, sb0, sw, carry, b + w.sub, ws_bytes - w.sub, st));
  } else {
    WT_TRY(wtconv_fwd(&c, ll, wb0, nullptr, wsub_c, sb0, sw, carry, b + w.sub, ws_bytes - w.sub, st));
  }
  e = wt::launch_add_carry(d->dtype, y, carry, (long long)d->N * d->C, d->H, d->W, s, st);
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "coarse-level split: %s", cudaGetErrorString(e));
  return ok();
}

// Parameter gradients of a split layer: the fine pass writes the base
// gradients and levels 1..s, the coarse layer levels s+1..L (its wavelet-scale
// gradient scaled by 4^-s afterwards).
wtconv_status_t split_bw(const wtconv_desc_t* d, int s, const void* x, const void* dy, const float* w_base,
                         const float* b_base, const float* w_sub, const float* base_scale,
                         const float* wavelet_scale, float* dw_base, float* db_base, float* dw_sub,
                         float* dbase_scale, float* dwavelet_scale, void* ws, size_t ws_bytes, cudaStream_t st) {
  const SplitLayout w = split_layout(d, WTCONV_OP_BWD_WEIGHT, s);
  WT_TRY(split_workspace_ok(w, ws, ws_bytes));
  const wtconv_desc_t f = fine_desc(d, s), c = coarse_desc(d, s);
  const size_t KK = (size_t)d->k * d->k, C = (size_t)d->C;
  char* b = static_cast<char*>(ws);
  float* llx = reinterpret_cast<float*>(b + w.ll);
  float* lld = reinterpret_cast<float*>(b + w.ll2);
  const float* wb0 = reinterpret_cast<const float*>(b + w.zeros);
  const float* sb0 = wb0 + C * KK;
  const float* sw = reinterpret_cast<const float*>(b + w.sw);
  float* dwb0 = reinterpret_cast<float*>(b + w.dummy);
  float* dsb0 = dwb0 + C * KK;
  WT_TRY(wtconv_bwd_weight(&f, x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, dw_base, db_base, dw_sub,
                           dbase_scale, dwavelet_scale, b + w.fine, w.fine_bytes, st));
  WT_TRY(split_params(d, s, wavelet_scale, b, w, st));
  cudaError_t e = wt::launch_lowpass(d->dtype, x, llx, (long long)d->N * d->C, d->H, d->W, s, st);
  if (e == cudaSuccess) e = wt::launch_lowpass(d->dtype, dy, lld, (long long)d->N * d->C, d->H, d->W, s, st);
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "coarse-level split: %s", cudaGetErrorString(e));
  float* dsw_c = dwavelet_scale + (size_t)s * 4 * C;
  WT_TRY(wtconv_bwd_weight(&c, llx, lld, wb0, nullptr, w_sub + (size_t)s * 4 * C * KK, sb0, sw, dwb0, nullptr,
                           dw_sub + (size_t)s * 4 * C * KK, dsb0, dsw_c, b + w.sub, ws_bytes - w.sub, st));
  e = wt::launch_scale(dsw_c, dsw_c, (d->levels - s) * 4 * d->C, ldexpf(1.f, -2 * s), st);
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "coarse-level split: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

namespace wt {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

namespace {
std::mutex g_cache_mu;
std::map<std::pair<int, const void*>, int> g_smem_set;                    // (device, kernel) -> limit set
std::map<std::tuple<int, const void*, int, int>, int> g_occupancy;        // (device, kernel, threads, smem)
std::map<int, int> g_sms;                                                 // device -> SM count
}  // namespace

cudaError_t ensure_smem(const void* f, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cache_mu);
  auto it = g_smem_set.find({dev, f});
  if (it != g_smem_set.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_smem_set[{dev, f}] = bytes;
  return e;
}

int occupancy(const void* f, int threads, int smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    auto it = g_occupancy.find({dev, f, threads, smem});
    if (it != g_occupancy.end()) return it->second;
  }
  int n = 0;
  if (ensure_smem(f, smem) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(g_cache_mu);
  g_occupancy[{dev, f, threads, smem}] = n;
  return n;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  {
    std::lock_guard<std::mutex> lock(g_cache_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) return it->second;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(g_cache_mu);
  g_sms[dev] = n;
  return n;
}
}  // namespace wt

extern "C" {

size_t wtconv_workspace_size(const wtconv_desc_t* desc, int op) {
  if (validate_desc(desc) != WTCONV_OK) return 0;
  if (op == WTCONV_OP_BWD) {
    WtBwPlan pl;
    WtFwdPlan fp;
    const wtconv_status_t st = plan_bwf(desc, pl, fp);
    if (st == WTCONV_OK) return bw_workspace_bytes(pl);
    if (st != WTCONV_ERR_UNSUPPORTED) return 0;
    // the call runs the two separate passes, one after the other, in the same workspace
    return std::max(wtconv_workspace_size(desc, WTCONV_OP_BWD_DATA),
                    wtconv_workspace_size(desc, WTCONV_OP_BWD_WEIGHT));
  }
  if (op == WTCONV_OP_FWD || op == WTCONV_OP_BWD_DATA) return split_bytes(desc, op);
  if (op != WTCONV_OP_BWD_WEIGHT) return 0;
  WtBwPlan pl;
  const wtconv_status_t st = plan_bw(desc, pl);
  if (st == WTCONV_OK) return bw_workspace_bytes(pl);
  if (st != WTCONV_ERR_UNSUPPORTED) return 0;
  // Windowed: the plan (and with it the grid and the record count) depends on
  // how the tensors can be loaded, which the pointers decide at call time;
  // the size covers every way.
  size_t bytes = 0;
  const int box = desc->dtype == WTCONV_F32 ? (desc->W % 4 == 0 ? 1 : 0) : (desc->W % 8 == 0 ? 2 : 0);
  for (int load = 0; load <= box; load += box > 0 ? box : 1) {
    if (plan_bw_win(desc, pl, load) == WTCONV_OK) bytes = std::max(bytes, bw_workspace_bytes(pl));
  }
  return std::max(bytes, split_bytes(desc, WTCONV_OP_BWD_WEIGHT));
}

wtconv_status_t wtconv_fwd(const wtconv_desc_t* desc, const void* x, const float* w_base,
                           const float* b_base, const float* w_sub, const float* base_scale,
                           const float* wavelet_scale, void* y, void* ws, size_t ws_bytes,
                           void* stream) {
  WT_TRY(validate_desc(desc));
  WT_TRY(check_param(w_base, "w_base", false));
  WT_TRY(check_param(b_base, "b_base", true));
  WT_TRY(check_param(w_sub, "w_sub", false));
  WT_TRY(check_param(base_scale, "base_scale", false));
  WT_TRY(check_param(wavelet_scale, "wavelet_scale", false));
  WtFwdPlan pl;
  const wtconv_status_t pst = plan_any(desc, pl, x);
  const int split = pst == WTCONV_ERR_UNSUPPORTED ? split_levels(desc, false) : 0;
  if (split == 0) WT_TRY(pst);
  if (desc->N == 0) return ok();
  if (split > 0)
    return split_fwd(desc, split, false, x, w_base, b_base, w_sub, base_scale, wavelet_scale, y, ws, ws_bytes,
                     (cudaStream_t)stream);
  WT_TRY(check_act(x, "x", desc));
  WT_TRY(check_act(y, "y", desc));
  alignas(64) CUtensorMap tmx;
  memset(&tmx, 0, sizeof(tmx));
  cudaError_t e;
  if (pl.win) {
    WT_TRY(prepare_win(desc, pl, &tmx, x, y));
    apply_wait_hook(pl);
    e = wt::launch_fwd_win(pl, tmx, desc->dtype, false, x, w_base, b_base, w_sub, base_scale, wavelet_scale, y,
                           (cudaStream_t)stream);
  } else {
    set_load_divs(pl, desc, vec_ok(desc, x, y));
    pl.use_tma = encode_plane_map(&tmx, x, desc, pl.lev[0].stride, pl.lev[0].band / pl.lev[0].stride, pl.P);
    set_bulk(pl, desc, x, 4L * (pl.work_off - pl.stage_off));
    apply_wait_hook(pl);
    e = wt::launch_fwd(pl, tmx, desc->dtype, false, x, w_base, b_base, w_sub, base_scale, wavelet_scale, y,
                       (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "wtconv_fwd: %s", cudaGetErrorString(e));
  return ok();
}

wtconv_status_t wtconv_bwd_data(const wtconv_desc_t* desc, const void* dy, const float* w_base,
                                const float* w_sub, const float* base_scale,
                                const float* wavelet_scale, void* dx, void* ws, size_t ws_bytes,
                                void* stream) {
  WT_TRY(validate_desc(desc));
  WT_TRY(check_param(w_base, "w_base", false));
  WT_TRY(check_param(w_sub, "w_sub", false));
  WT_TRY(check_param(base_scale, "base_scale", false));
  WT_TRY(check_param(wavelet_scale, "wavelet_scale", false));
  WtFwdPlan pl;
  const wtconv_status_t pst = plan_any(desc, pl, dy);
  const int split = pst == WTCONV_ERR_UNSUPPORTED ? split_levels(desc, false) : 0;
  if (split == 0) WT_TRY(pst);
  if (desc->N == 0) return ok();
  if (split > 0)
    return split_fwd(desc, split, true, dy, w_base, nullptr, w_sub, base_scale, wavelet_scale, dx, ws, ws_bytes,
                     (cudaStream_t)stream);
  WT_TRY(check_act(dy, "dy", desc));
  WT_TRY(check_act(dx, "dx", desc));
  alignas(64) CUtensorMap tmx;
  memset(&tmx, 0, sizeof(tmx));
  cudaError_t e;
  if (pl.win) {
    WT_TRY(prepare_win(desc, pl, &tmx, dy, dx));
    apply_wait_hook(pl);
    e = wt::launch_fwd_win(pl, tmx, desc->dtype, true, dy, w_base, nullptr, w_sub, base_scale, wavelet_scale,
                           dx, (cudaStream_t)stream);
  } else {
    set_load_divs(pl, desc, vec_ok(desc, dy, dx));
    pl.use_tma = encode_plane_map(&tmx, dy, desc, pl.lev[0].stride, pl.lev[0].band / pl.lev[0].stride, pl.P);
    set_bulk(pl, desc, dy, 4L * (pl.work_off - pl.stage_off));
    apply_wait_hook(pl);
    e = wt::launch_fwd(pl, tmx, desc->dtype, true, dy, w_base, nullptr, w_sub, base_scale, wavelet_scale, dx,
                       (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "wtconv_bwd_data: %s", cudaGetErrorString(e));
  return ok();
}

wtconv_status_t wtconv_bwd(const wtconv_desc_t* desc, const void* x, const void* dy, const float* w_base,
                           const float* b_base, const float* w_sub, const float* base_scale,
                           const float* wavelet_scale, void* dx, float* dw_base, float* db_base, float* dw_sub,
                           float* dbase_scale, float* dwavelet_scale, void* ws, size_t ws_bytes, void* stream) {
  WT_TRY(validate_desc(desc));
  WT_TRY(check_param(w_base, "w_base", false));
  WT_TRY(check_param(b_base, "b_base", true));
  WT_TRY(check_param(w_sub, "w_sub", false));
  WT_TRY(check_param(base_scale, "base_scale", false));
  WT_TRY(check_param(wavelet_scale, "wavelet_scale", false));
  WT_TRY(check_param(dw_base, "dw_base", false));
  WT_TRY(check_param(db_base, "db_base", true));
  WT_TRY(check_param(dw_sub, "dw_sub", false));
  WT_TRY(check_param(dbase_scale, "dbase_scale", false));
  WT_TRY(check_param(dwavelet_scale, "dwavelet_scale", false));
  WtBwPlan pl;
  WtFwdPlan fp;
  const wtconv_status_t st = plan_bwf(desc, pl, fp);
  if (st == WTCONV_ERR_UNSUPPORTED || desc->N == 0) {
    // Planes beyond the fused kernel's working set (or an empty batch): the
    // two separate passes, with the same results.
    WT_TRY(wtconv_bwd_data(desc, dy, w_base, w_sub, base_scale, wavelet_scale, dx, ws, ws_bytes, stream));
    return wtconv_bwd_weight(desc, x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, dw_base, db_base,
                             dw_sub, dbase_scale, dwavelet_scale, ws, ws_bytes, stream);
  }
  if (st != WTCONV_OK) return st;
  WT_TRY(check_act(x, "x", desc));
  WT_TRY(check_act(dy, "dy", desc));
  WT_TRY(check_act(dx, "dx", desc));
  const size_t need = bw_workspace_bytes(pl);
  if (!ws || ws_bytes < need)
    return fail(WTCONV_ERR_WORKSPACE, "workspace of %zu B given, %zu B needed", ws ? ws_bytes : 0, need);
  if (!aligned(ws, 256)) return fail(WTCONV_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  set_load_divs(pl, desc, vec_ok(desc, x, dy));
  fp.vec_ok = vec_ok(desc, dx, nullptr);
  set_bulk(pl, desc, x, pl.work_off > pl.stage_off ? 4L * (pl.work_off - pl.stage_off) / 2 : 0);
  if (pl.use_bulk == 1 && !(aligned(dy, 16) && 2L * pl.P * pl.bulk_bytes < (1L << 20))) pl.use_bulk = 2;
  if (pl.use_bulk == 2 && !aligned(dy, 8)) pl.use_bulk = 0;
  alignas(64) CUtensorMap tmx, tmd;
  memset(&tmx, 0, sizeof(tmx));
  memset(&tmd, 0, sizeof(tmd));
  pl.use_tma = encode_plane_map(&tmx, x, desc, pl.xs[0].stride, pl.xbf / pl.xs[0].stride, pl.P) &&
               encode_plane_map(&tmd, dy, desc, pl.ds[0].stride, pl.dbf / pl.ds[0].stride, pl.P);
  apply_wait_hook(pl);
  cudaError_t e = wt::launch_bwd_fused(pl, fp, tmx, tmd, desc->dtype, x, dy, w_base, b_base, w_sub, base_scale,
                                       wavelet_scale, dx, dw_base, db_base, dw_sub, dbase_scale, dwavelet_scale,
                                       static_cast<float*>(ws), (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "wtconv_bwd: %s", cudaGetErrorString(e));
  return ok();
}

wtconv_status_t wtconv_bwd_weight(const wtconv_desc_t* desc, const void* x, const void* dy,
                                  const float* w_base, const float* b_base, const float* w_sub,
                                  const float* base_scale, const float* wavelet_scale,
                                  float* dw_base, float* db_base, float* dw_sub, float* dbase_scale,
                                  float* dwavelet_scale, void* ws, size_t ws_bytes, void* stream) {
  WT_TRY(validate_desc(desc));
  WT_TRY(check_param(w_base, "w_base", false));
  WT_TRY(check_param(b_base, "b_base", true));
  WT_TRY(check_param(w_sub, "w_sub", false));
  WT_TRY(check_param(base_scale, "base_scale", false));
  WT_TRY(check_param(wavelet_scale, "wavelet_scale", false));
  WT_TRY(check_param(dw_base, "dw_base", false));
  WT_TRY(check_param(db_base, "db_base", true));
  WT_TRY(check_param(dw_sub, "dw_sub", false));
  WT_TRY(check_param(dbase_scale, "dbase_scale", false));
  WT_TRY(check_param(dwavelet_scale, "dwavelet_scale", false));
  WtBwPlan pl;
  const wtconv_status_t pst = plan_bw_any(desc, pl, x, dy);
  const int split = pst == WTCONV_ERR_UNSUPPORTED ? split_levels(desc, true) : 0;
  if (split == 0) WT_TRY(pst);
  cudaStream_t st = (cudaStream_t)stream;
  const int C = desc->C, L = desc->levels, KK = desc->k * desc->k;
  if (desc->N == 0) {  // empty batch: every gradient is an empty sum
    cudaError_t e = cudaMemsetAsync(dw_base, 0, sizeof(float) * C * KK, st);
    if (e == cudaSuccess && db_base) e = cudaMemsetAsync(db_base, 0, sizeof(float) * C, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dw_sub, 0, sizeof(float) * (size_t)L * 4 * C * KK, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dbase_scale, 0, sizeof(float) * C, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(dwavelet_scale, 0, sizeof(float) * (size_t)L * 4 * C, st);
    if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "wtconv_bwd_weight: %s", cudaGetErrorString(e));
    return ok();
  }
  if (split > 0)
    return split_bw(desc, split, x, dy, w_base, b_base, w_sub, base_scale, wavelet_scale, dw_base, db_base, dw_sub,
                    dbase_scale, dwavelet_scale, ws, ws_bytes, st);
  WT_TRY(check_act(x, "x", desc));
  WT_TRY(check_act(dy, "dy", desc));
  alignas(64) CUtensorMap tmx, tmd;
  memset(&tmx, 0, sizeof(tmx));
  memset(&tmd, 0, sizeof(tmd));
  if (pl.win) {
    // box copies of the x windows and dy tiles (re-planned for plain loads if
    // a map cannot be encoded), then the plain-load divisors
    bool boxed = true;
    if (pl.win_load == 1)
      boxed = encode_plane_map(&tmx, x, desc, pl.xs[0].stride, pl.xbf / pl.xs[0].stride, pl.P) &&
              encode_plane_map(&tmd, dy, desc, pl.ds[0].stride, pl.th, pl.P);
    else if (pl.win_load == 2)
      boxed = encode_map16(&tmx, x, desc, pl.Ws[0], pl.Hs[0], pl.P) &&
              encode_map16(&tmd, dy, desc, pl.tw, pl.th, pl.P);
    if (!boxed) WT_TRY(plan_bw_win(desc, pl, 0));
    pl.vec_ok = vec_ok(desc, x, dy);
    const int v = pl.vec_ok ? (int)(16 / elem_size(desc->dtype)) : 1;
    pl.ld_pp = make_div(pl.Hs[0] * (pl.Ws[0] / v));
    pl.ld_w = make_div(pl.Ws[0] / v);
    pl.dld_pp = make_div(pl.th * (pl.tw / v));
    pl.dld_w = make_div(pl.tw / v);
  }
  const size_t need = bw_workspace_bytes(pl);
  if (!ws || ws_bytes < need)
    return fail(WTCONV_ERR_WORKSPACE, "workspace of %zu B given, %zu B needed", ws ? ws_bytes : 0, need);
  if (!aligned(ws, 256)) return fail(WTCONV_ERR_MISALIGNED, "workspace is not 256-byte aligned");
  if (pl.win) {
    apply_wait_hook(pl);
    cudaError_t e = wt::launch_bwd_weight_win(pl, tmx, tmd, desc->dtype, x, dy, w_base, b_base, w_sub, base_scale,
                                              wavelet_scale, dw_base, db_base, dw_sub, dbase_scale, dwavelet_scale,
                                              static_cast<float*>(ws), st);
    if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "wtconv_bwd_weight: %s", cudaGetErrorString(e));
    return ok();
  }
  set_load_divs(pl, desc, vec_ok(desc, x, dy));
  set_bulk(pl, desc, x, pl.stage_off > 0 ? 4L * (pl.work_off - pl.stage_off) / 2 : 0);
  if (pl.use_bulk == 1 && !(aligned(dy, 16) && 2L * pl.P * pl.bulk_bytes < (1L << 20))) pl.use_bulk = 2;
  if (pl.use_bulk == 2 && !aligned(dy, 8)) pl.use_bulk = 0;
  pl.use_tma = encode_plane_map(&tmx, x, desc, pl.xs[0].stride, pl.xbf / pl.xs[0].stride, pl.P) &&
               encode_plane_map(&tmd, dy, desc, pl.ds[0].stride, pl.dbf / pl.ds[0].stride, pl.P);
  apply_wait_hook(pl);
  cudaError_t e = wt::launch_bwd_weight(pl, tmx, tmd, desc->dtype, x, dy, w_base, b_base, w_sub, base_scale,
                                        wavelet_scale, dw_base, db_base, dw_sub, dbase_scale,
                                        dwavelet_scale, static_cast<float*>(ws), st);
  if (e != cudaSuccess) return fail(WTCONV_ERR_CUDA, "wtconv_bwd_weight: %s", cudaGetErrorString(e));
  return ok();
}

const char* wtconv_status_string(wtconv_status_t s) {
  switch (s) {
    case WTCONV_OK: return "WTCONV_OK";
    case WTCONV_ERR_INVALID_ARG: return "WTCONV_ERR_INVALID_ARG";
    case WTCONV_ERR_UNSUPPORTED: return "WTCONV_ERR_UNSUPPORTED";
    case WTCONV_ERR_MISALIGNED: return "WTCONV_ERR_MISALIGNED";
    case WTCONV_ERR_WORKSPACE: return "WTCONV_ERR_WORKSPACE";
    case WTCONV_ERR_CUDA: return "WTCONV_ERR_CUDA";
  }
  return "WTCONV_STATUS_UNKNOWN";
}

const char* wtconv_last_error(void) { return g_last_error; }

void wtconv_test_copy_timeout(int enable) {
  std::lock_guard<std::mutex> lock(g_hook_mu);
  g_hook_on = enable != 0;
}

unsigned int wtconv_device_faults(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return 0;
  return wt::take_fwd_faults() + wt::take_win_faults() + wt::take_bw_faults() + wt::take_bww_faults() +
         wt::take_bwf_faults();
}

}  // extern "C"
