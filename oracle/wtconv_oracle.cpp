// WTConv2d CPU oracle -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, float64 statement of the WTConv2d layer (forward and
// backward).  Only the test suite, the smoke check and the benchmark's CPU
// baseline use it; the product path never links, loads or calls it.  It
// shares no code, header or constant with the CUDA library.
//
// Source of the definition: "Fast and Memory-Efficient Wavelet Convolutions
// via I/O-Aware Reformulation" (Aflalo, Finder, Amoyal, Treister, Freifeld;
// arXiv 2608.10805), as given by its abstract (arxivdaily page) and by the
// technical summary on gist.science (sections "Problem statement",
// "Methodology", "Key contributions").  Citations below name the section.
//
// The layer (technical summary, "Methodology": the reference implementation
// runs a Haar analysis pass, a depthwise convolution per subband, a learned
// per-channel scale as a separate elementwise pass, an L-step synthesis loop in
// which each level adds the previous reconstruction to the low-pass subband
// and applies a transposed convolution, plus a scaled base depthwise
// convolution with a bias):
//
//   cur = x
//   for l = 1..L:  Y^l = Haar(pad_even(cur));  Z^l_b = s_w[l,4c+b] * conv(Y^l_b, W_l[4c+b]);  cur = Y^l_0
//   next = 0
//   for l = L..1:  next = crop(Haar^T(Z^l + [next in band 0]))
//   y = s_base[c] * (conv(x, W_base[c]) + b[c]) + next
//
// Readings taken where the pages are silent (each also listed in the design
// notes): orthonormal Haar taps +-1/2; band order b = 0 LL, 1 row-high (sign
// (-1)^u for row offset u), 2 column-high (sign (-1)^v), 3 diagonal
// ((-1)^(u+v)); subband channel 4c+b; one wavelet scale per subband channel;
// the *unconvolved* LL feeds the next level; odd sizes are zero-padded on the
// bottom/right before each analysis and cropped after each synthesis;
// convolutions are stride-1 cross-correlations with zero "same" padding,
// k odd; the bias sits on the base path only and is multiplied by the base
// scale.
//
// Two independent forms are provided:
//   Form A ("cascade"): the unfused stages above, run in the pages' order,
//     with a hand-written adjoint of each stage for the backward pass.
//   Form B ("direct"):  each level's coefficients as a direct block sum over
//     the input, the synthesis as the closed-form bit-indexed sum
//     (technical summary, "Methodology", collapse of the multi-level synthesis
//     cascade, "Proposition 2"), dx as the brute-force transpose of the
//     assembled operator, parameter gradients as explicit correlation sums.
//     Only meant for tiny shapes.
//
// Parity status: every function here is pinned by tests that do not call
// this file's arithmetic twice (perfect reconstruction, Parseval, closed
// forms for delta kernels, single-band projections, torch library
// compositions with autograd, linearity, the adjoint identity, finite
// differences, Form A == Form B).

#include <cmath>
#include <cstddef>
#include <cstring>
#include <vector>

namespace {

typedef std::vector<double> Vec;

// sigma_b(u, v): sign of Haar band b at row offset u, column offset v.
double band_sign(int b, int u, int v) {
  int parity = 0;
  if (b == 1) parity = u;
  else if (b == 2) parity = v;
  else if (b == 3) parity = u + v;
  return (parity & 1) ? -1.0 : 1.0;
}

int half_up(int n) { return (n + 1) / 2; }

// One level of orthonormal 2D Haar analysis of an H x W plane, zero-padded
// on the bottom/right to even size.  out: [4][Hh][Wh].
void haar_analysis(const double* in, int H, int W, double* out) {
  const int Hh = half_up(H), Wh = half_up(W);
  for (int b = 0; b < 4; ++b)
    for (int p = 0; p < Hh; ++p)
      for (int q = 0; q < Wh; ++q) {
        double s = 0.0;
        for (int u = 0; u < 2; ++u)
          for (int v = 0; v < 2; ++v) {
            const int i = 2 * p + u, j = 2 * q + v;
            const double val = (i < H && j < W) ? in[(size_t)i * W + j] : 0.0;
            s += band_sign(b, u, v) * val;
          }
        out[((size_t)b * Hh + p) * Wh + q] = 0.5 * s;
      }
}

// One level of Haar synthesis (the transpose of haar_analysis): 4 bands of
// Hh x Wh -> a 2Hh x 2Wh plane, cropped to H x W.
void haar_synthesis(const double* in, int Hh, int Wh, double* out, int H, int W) {
  for (int i = 0; i < H; ++i)
    for (int j = 0; j < W; ++j) {
      const int p = i / 2, u = i % 2, q = j / 2, v = j % 2;
      double s = 0.0;
      for (int b = 0; b < 4; ++b) s += band_sign(b, u, v) * in[((size_t)b * Hh + p) * Wh + q];
      out[(size_t)i * W + j] = 0.5 * s;
    }
}

// Stride-1 depthwise cross-correlation with zero "same" padding (k odd).
void conv_same(const double* in, int H, int W, const double* w, int K, double* out) {
  const int r = K / 2;
  for (int i = 0; i < H; ++i)
    for (int j = 0; j < W; ++j) {
      double s = 0.0;
      for (int du = 0; du < K; ++du)
        for (int dv = 0; dv < K; ++dv) {
          const int ii = i + du - r, jj = j + dv - r;
          if (ii >= 0 && ii < H && jj >= 0 && jj < W) s += w[du * K + dv] * in[(size_t)ii * W + jj];
        }
      out[(size_t)i * W + j] = s;
    }
}

// Adjoint of conv_same with respect to its input: out += conv_same^T(g).
void conv_same_adjoint_add(const double* g, int H, int W, const double* w, int K, double scale,
                           double* out) {
  const int r = K / 2;
  for (int i = 0; i < H; ++i)
    for (int j = 0; j < W; ++j) {
      const double gv = scale * g[(size_t)i * W + j];
      for (int du = 0; du < K; ++du)
        for (int dv = 0; dv < K; ++dv) {
          const int ii = i + du - r, jj = j + dv - r;
          if (ii >= 0 && ii < H && jj >= 0 && jj < W) out[(size_t)ii * W + jj] += w[du * K + dv] * gv;
        }
    }
}

// Gradient of conv_same with respect to its weights: G[t] += sum g[i,j] * in[i+du-r, j+dv-r].
void conv_same_weight_grad_add(const double* g, const double* in, int H, int W, int K, double* G) {
  const int r = K / 2;
  for (int du = 0; du < K; ++du)
    for (int dv = 0; dv < K; ++dv) {
      double s = 0.0;
      for (int i = 0; i < H; ++i)
        for (int j = 0; j < W; ++j) {
          const int ii = i + du - r, jj = j + dv - r;
          if (ii >= 0 && ii < H && jj >= 0 && jj < W) s += g[(size_t)i * W + j] * in[(size_t)ii * W + jj];
        }
      G[du * K + dv] += s;
    }
}

double dot(const double* a, const double* b, size_t n) {
  double s = 0.0;
  for (size_t i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

struct Geometry {
  int H, W, L, K;
  std::vector<int> Hs, Ws;  // Hs[l], Ws[l] for l = 0..L
  Geometry(int H_, int W_, int L_, int K_) : H(H_), W(W_), L(L_), K(K_), Hs(L_ + 1), Ws(L_ + 1) {
    Hs[0] = H;
    Ws[0] = W;
    for (int l = 1; l <= L; ++l) {
      Hs[l] = half_up(Hs[l - 1]);
      Ws[l] = half_up(Ws[l - 1]);
    }
  }
  size_t plane(int l) const { return (size_t)Hs[l] * Ws[l]; }
};

bool valid_args(int N, int C, int H, int W, int L, int K) {
  return N >= 0 && C >= 1 && H >= 1 && W >= 1 && L >= 1 && L <= 16 && K >= 1 && (K % 2) == 1;
}

// Parameter views for channel c.
struct Params {
  const double* w_base;         // [C,K,K]
  const double* b_base;         // [C] or null
  const double* w_sub;          // [L,4C,K,K]
  const double* base_scale;     // [C]
  const double* wavelet_scale;  // [L,4C]
  int C, K;
  const double* wb(int c) const { return w_base + (size_t)c * K * K; }
  double bias(int c) const { return b_base ? b_base[c] : 0.0; }
  const double* ws(int l, int c, int b) const {  // level l in 1..L
    return w_sub + (((size_t)(l - 1) * 4 * C) + 4 * c + b) * K * K;
  }
  double sw(int l, int c, int b) const { return wavelet_scale[(size_t)(l - 1) * 4 * C + 4 * c + b]; }
};

// ---------------------------------------------------------------- Form A --

// Forward of one (n, c) plane, unfused cascade.
void fwd_plane_cascade(const Geometry& g, const Params& P, int c, const double* x, double* y) {
  const int L = g.L, K = g.K;
  std::vector<Vec> Z(L + 1);
  Vec cur(x, x + g.plane(0));
  for (int l = 1; l <= L; ++l) {
    Vec Y(4 * g.plane(l));
    haar_analysis(cur.data(), g.Hs[l - 1], g.Ws[l - 1], Y.data());
    Z[l].assign(4 * g.plane(l), 0.0);
    for (int b = 0; b < 4; ++b) {
      double* zb = Z[l].data() + b * g.plane(l);
      conv_same(Y.data() + b * g.plane(l), g.Hs[l], g.Ws[l], P.ws(l, c, b), K, zb);
      const double s = P.sw(l, c, b);
      for (size_t t = 0; t < g.plane(l); ++t) zb[t] *= s;  // the separate scale pass
    }
    cur.assign(Y.begin(), Y.begin() + g.plane(l));  // unconvolved LL feeds the next level
  }
  Vec next(g.plane(L), 0.0);
  for (int l = L; l >= 1; --l) {
    Vec Zl = Z[l];
    for (size_t t = 0; t < g.plane(l); ++t) Zl[t] += next[t];  // add previous reconstruction to LL
    Vec out(g.plane(l - 1));
    haar_synthesis(Zl.data(), g.Hs[l], g.Ws[l], out.data(), g.Hs[l - 1], g.Ws[l - 1]);
    next.swap(out);
  }
  Vec base(g.plane(0));
  conv_same(x, g.H, g.W, P.wb(c), K, base.data());
  const double sb = P.base_scale[c], bias = P.bias(c);
  for (size_t t = 0; t < g.plane(0); ++t) y[t] = sb * (base[t] + bias) + next[t];
}

// Backward of one (n, c) plane: hand-written adjoint of each stage, in
// reverse order.  Parameter gradients are accumulated (+=).
void bwd_plane_cascade(const Geometry& g, const Params& P, int c, const double* x, const double* dy,
                       double* dx, double* dw_base, double* db, double* dw_sub_c /*[L][4][K*K]*/,
                       double* dsb, double* dsw_c /*[L][4]*/) {
  const int L = g.L, K = g.K, KK = K * K;
  // recompute the forward intermediates
  std::vector<Vec> Y(L + 1), Cv(L + 1);
  Vec cur(x, x + g.plane(0));
  for (int l = 1; l <= L; ++l) {
    Y[l].assign(4 * g.plane(l), 0.0);
    haar_analysis(cur.data(), g.Hs[l - 1], g.Ws[l - 1], Y[l].data());
    Cv[l].assign(4 * g.plane(l), 0.0);
    for (int b = 0; b < 4; ++b)
      conv_same(Y[l].data() + b * g.plane(l), g.Hs[l], g.Ws[l], P.ws(l, c, b), K,
                Cv[l].data() + b * g.plane(l));
    cur.assign(Y[l].begin(), Y[l].begin() + g.plane(l));
  }
  // base path: y_base = s * (conv(x, W) + b)
  const double sb = P.base_scale[c];
  Vec Gb(KK, 0.0);
  conv_same_weight_grad_add(dy, x, g.H, g.W, K, Gb.data());
  double gsum = 0.0;
  for (size_t t = 0; t < g.plane(0); ++t) gsum += dy[t];
  for (int t = 0; t < KK; ++t) dw_base[t] += sb * Gb[t];
  if (db) *db += sb * gsum;
  *dsb += dot(P.wb(c), Gb.data(), KK) + P.bias(c) * gsum;
  Vec dxv(g.plane(0), 0.0);
  conv_same_adjoint_add(dy, g.H, g.W, P.wb(c), K, sb, dxv.data());
  // synthesis cascade adjoint: crop^T then synthesis^T = zero-pad then analysis
  std::vector<Vec> gY(L + 1);
  Vec gnext(dy, dy + g.plane(0));
  for (int l = 1; l <= L; ++l) {
    Vec gZ(4 * g.plane(l));
    haar_analysis(gnext.data(), g.Hs[l - 1], g.Ws[l - 1], gZ.data());
    gY[l].assign(4 * g.plane(l), 0.0);
    for (int b = 0; b < 4; ++b) {
      const double* gzb = gZ.data() + b * g.plane(l);
      const double s = P.sw(l, c, b);
      Vec G(KK, 0.0);
      conv_same_weight_grad_add(gzb, Y[l].data() + b * g.plane(l), g.Hs[l], g.Ws[l], K, G.data());
      for (int t = 0; t < KK; ++t) dw_sub_c[((size_t)(l - 1) * 4 + b) * KK + t] += s * G[t];
      dsw_c[(l - 1) * 4 + b] += dot(gzb, Cv[l].data() + b * g.plane(l), g.plane(l));
      conv_same_adjoint_add(gzb, g.Hs[l], g.Ws[l], P.ws(l, c, b), K, s, gY[l].data() + b * g.plane(l));
    }
    gnext.assign(gZ.begin(), gZ.begin() + g.plane(l));  // gradient w.r.t. next^l (added into LL)
  }
  // analysis chain adjoint: LL^l = Y^l_0 feeds level l+1
  Vec acc(g.plane(L), 0.0);
  for (int l = L; l >= 1; --l) {
    Vec gYt = gY[l];
    for (size_t t = 0; t < g.plane(l); ++t) gYt[t] += acc[t];
    Vec out(g.plane(l - 1));
    haar_synthesis(gYt.data(), g.Hs[l], g.Ws[l], out.data(), g.Hs[l - 1], g.Ws[l - 1]);
    acc.swap(out);
  }
  for (size_t t = 0; t < g.plane(0); ++t) dx[t] = dxv[t] + acc[t];
}

// ---------------------------------------------------------------- Form B --

// Zero-extended input.
double xt(const double* x, int H, int W, long i, long j) {
  return (i >= 0 && i < H && j >= 0 && j < W) ? x[(size_t)i * W + j] : 0.0;
}

int bit(long v, int k) { return (int)((v >> k) & 1); }

// Level-l coefficients as a direct block sum over the zero-extended input:
// Y^l_b[p,q] = 0.5^l * sum_{u,v < 2^l} sigma_b(bit_{l-1}(u), bit_{l-1}(v)) x~[2^l p + u, 2^l q + v].
void direct_coefficients(const double* x, int H, int W, int l, int Hl, int Wl, double* Y) {
  const long S = 1L << l;
  const double norm = std::ldexp(1.0, -l);
  for (int b = 0; b < 4; ++b)
    for (int p = 0; p < Hl; ++p)
      for (int q = 0; q < Wl; ++q) {
        double s = 0.0;
        for (long u = 0; u < S; ++u)
          for (long v = 0; v < S; ++v)
            s += band_sign(b, bit(u, l - 1), bit(v, l - 1)) * xt(x, H, W, S * p + u, S * q + v);
        Y[((size_t)b * Hl + p) * Wl + q] = norm * s;
      }
}

// Explicit tap loop, zero outside [0,H) x [0,W).
double tap_sum(const double* in, int H, int W, const double* w, int K, int i, int j) {
  const int r = K / 2;
  double s = 0.0;
  for (int du = 0; du < K; ++du)
    for (int dv = 0; dv < K; ++dv) s += w[du * K + dv] * xt(in, H, W, i + du - r, j + dv - r);
  return s;
}

void fwd_plane_direct(const Geometry& g, const Params& P, int c, const double* x, double* y,
                      bool with_bias) {
  const int L = g.L, K = g.K;
  std::vector<Vec> Z(L + 1);
  for (int l = 1; l <= L; ++l) {
    Vec Y(4 * g.plane(l));
    direct_coefficients(x, g.H, g.W, l, g.Hs[l], g.Ws[l], Y.data());
    Z[l].assign(4 * g.plane(l), 0.0);
    for (int b = 0; b < 4; ++b)
      for (int p = 0; p < g.Hs[l]; ++p)
        for (int q = 0; q < g.Ws[l]; ++q)
          Z[l][((size_t)b * g.Hs[l] + p) * g.Ws[l] + q] =
              P.sw(l, c, b) * tap_sum(Y.data() + b * g.plane(l), g.Hs[l], g.Ws[l], P.ws(l, c, b), K, p, q);
  }
  const double bias = with_bias ? P.bias(c) : 0.0;
  for (int i = 0; i < g.H; ++i)
    for (int j = 0; j < g.W; ++j) {
      double acc = P.base_scale[c] * (tap_sum(x, g.H, g.W, P.wb(c), K, i, j) + bias);
      // closed-form bit-indexed synthesis
      for (int l = 1; l <= L; ++l) {
        const int u = bit(i, l - 1), v = bit(j, l - 1);
        const int p = i >> l, q = j >> l;
        double s = 0.0;
        for (int b = 0; b < 4; ++b) s += band_sign(b, u, v) * Z[l][((size_t)b * g.Hs[l] + p) * g.Ws[l] + q];
        acc += std::ldexp(1.0, -l) * s;
      }
      y[(size_t)i * g.W + j] = acc;
    }
}

void bwd_plane_direct(const Geometry& g, const Params& P, int c, const double* x, const double* dy,
                      double* dx, double* dw_base, double* db, double* dw_sub_c, double* dsb,
                      double* dsw_c) {
  const int L = g.L, K = g.K, KK = K * K, r = K / 2;
  const size_t n0 = g.plane(0);
  // dx = A^T dy with A assembled column by column from unit impulses (bias off)
  Vec e(n0, 0.0), col(n0);
  for (size_t m = 0; m < n0; ++m) {
    e[m] = 1.0;
    fwd_plane_direct(g, P, c, e.data(), col.data(), false);
    e[m] = 0.0;
    dx[m] = dot(col.data(), dy, n0);
  }
  // base parameters: y_base = s * (sum_t W_t x~[i+t] + b)
  double gsum = 0.0;
  for (size_t t = 0; t < n0; ++t) gsum += dy[t];
  for (int du = 0; du < K; ++du)
    for (int dv = 0; dv < K; ++dv) {
      double G = 0.0;
      for (int i = 0; i < g.H; ++i)
        for (int j = 0; j < g.W; ++j) G += dy[(size_t)i * g.W + j] * xt(x, g.H, g.W, i + du - r, j + dv - r);
      dw_base[du * K + dv] += P.base_scale[c] * G;
      *dsb += P.wb(c)[du * K + dv] * G;
    }
  *dsb += P.bias(c) * gsum;
  if (db) *db += P.base_scale[c] * gsum;
  // wavelet parameters: dL/dZ^l = level-l coefficients of dy (same direct sum applied to dy)
  for (int l = 1; l <= L; ++l) {
    const int Hl = g.Hs[l], Wl = g.Ws[l];
    Vec Y(4 * g.plane(l)), D(4 * g.plane(l));
    direct_coefficients(x, g.H, g.W, l, Hl, Wl, Y.data());
    direct_coefficients(dy, g.H, g.W, l, Hl, Wl, D.data());
    for (int b = 0; b < 4; ++b) {
      const double* Yb = Y.data() + b * g.plane(l);
      const double* Db = D.data() + b * g.plane(l);
      for (int du = 0; du < K; ++du)
        for (int dv = 0; dv < K; ++dv) {
          double G = 0.0;
          for (int p = 0; p < Hl; ++p)
            for (int q = 0; q < Wl; ++q) G += Db[(size_t)p * Wl + q] * xt(Yb, Hl, Wl, p + du - r, q + dv - r);
          dw_sub_c[((size_t)(l - 1) * 4 + b) * KK + du * K + dv] += P.sw(l, c, b) * G;
          dsw_c[(l - 1) * 4 + b] += P.ws(l, c, b)[du * K + dv] * G;
        }
    }
  }
}

// ------------------------------------------------------------- drivers --

typedef void (*FwdPlaneFn)(const Geometry&, const Params&, int, const double*, double*);

void fwd_direct_with_bias(const Geometry& g, const Params& P, int c, const double* x, double* y) {
  fwd_plane_direct(g, P, c, x, y, true);
}

int run_fwd(FwdPlaneFn fn, int N, int C, int H, int W, int L, int K, const double* x,
            const double* w_base, const double* b_base, const double* w_sub, const double* base_scale,
            const double* wavelet_scale, double* y) {
  if (!valid_args(N, C, H, W, L, K)) return -1;
  Geometry g(H, W, L, K);
  Params P{w_base, b_base, w_sub, base_scale, wavelet_scale, C, K};
  for (int n = 0; n < N; ++n)
    for (int c = 0; c < C; ++c) {
      const size_t off = ((size_t)n * C + c) * g.plane(0);
      fn(g, P, c, x + off, y + off);
    }
  return 0;
}

typedef void (*BwdPlaneFn)(const Geometry&, const Params&, int, const double*, const double*, double*,
                           double*, double*, double*, double*, double*);

int run_bwd(BwdPlaneFn fn, int N, int C, int H, int W, int L, int K, const double* x, const double* dy,
            const double* w_base, const double* b_base, const double* w_sub, const double* base_scale,
            const double* wavelet_scale, double* dx, double* dw_base, double* db_base, double* dw_sub,
            double* dbase_scale, double* dwavelet_scale) {
  if (!valid_args(N, C, H, W, L, K)) return -1;
  Geometry g(H, W, L, K);
  Params P{w_base, b_base, w_sub, base_scale, wavelet_scale, C, K};
  const int KK = K * K;
  std::memset(dw_base, 0, sizeof(double) * C * KK);
  if (db_base) std::memset(db_base, 0, sizeof(double) * C);
  std::memset(dw_sub, 0, sizeof(double) * (size_t)L * 4 * C * KK);
  std::memset(dbase_scale, 0, sizeof(double) * C);
  std::memset(dwavelet_scale, 0, sizeof(double) * (size_t)L * 4 * C);
  Vec dws_c((size_t)L * 4 * KK), dsw_c((size_t)L * 4);
  for (int c = 0; c < C; ++c) {
    std::fill(dws_c.begin(), dws_c.end(), 0.0);
    std::fill(dsw_c.begin(), dsw_c.end(), 0.0);
    for (int n = 0; n < N; ++n) {
      const size_t off = ((size_t)n * C + c) * g.plane(0);
      fn(g, P, c, x + off, dy + off, dx + off, dw_base + (size_t)c * KK, db_base ? db_base + c : nullptr,
         dws_c.data(), dbase_scale + c, dsw_c.data());
    }
    for (int l = 1; l <= L; ++l)
      for (int b = 0; b < 4; ++b) {
        const size_t ch = (size_t)(l - 1) * 4 * C + 4 * c + b;
        for (int t = 0; t < KK; ++t) dw_sub[ch * KK + t] = dws_c[((size_t)(l - 1) * 4 + b) * KK + t];
        dwavelet_scale[ch] = dsw_c[(l - 1) * 4 + b];
      }
  }
  return 0;
}

}  // namespace

extern "C" {

// One level of Haar analysis (pad to even, 2x2 stride-2 butterfly, taps +-1/2).
void oracle_haar_analysis(const double* in, int H, int W, double* out) { haar_analysis(in, H, W, out); }

// One level of Haar synthesis with crop to H x W (transpose of the analysis).
void oracle_haar_synthesis(const double* in, int Hh, int Wh, double* out, int H, int W) {
  haar_synthesis(in, Hh, Wh, out, H, W);
}

// Form A forward.  Arrays are float64, C-contiguous; b_base may be null.
int oracle_fwd_cascade(int N, int C, int H, int W, int L, int K, const double* x, const double* w_base,
                       const double* b_base, const double* w_sub, const double* base_scale,
                       const double* wavelet_scale, double* y) {
  return run_fwd(fwd_plane_cascade, N, C, H, W, L, K, x, w_base, b_base, w_sub, base_scale,
                 wavelet_scale, y);
}

// Form B forward (direct sums; tiny shapes).
int oracle_fwd_direct(int N, int C, int H, int W, int L, int K, const double* x, const double* w_base,
                      const double* b_base, const double* w_sub, const double* base_scale,
                      const double* wavelet_scale, double* y) {
  return run_fwd(fwd_direct_with_bias, N, C, H, W, L, K, x, w_base, b_base, w_sub, base_scale,
                 wavelet_scale, y);
}

// Form A backward: dx and every parameter gradient (overwritten, not accumulated).
int oracle_bwd_cascade(int N, int C, int H, int W, int L, int K, const double* x, const double* dy,
                       const double* w_base, const double* b_base, const double* w_sub,
                       const double* base_scale, const double* wavelet_scale, double* dx, double* dw_base,
                       double* db_base, double* dw_sub, double* dbase_scale, double* dwavelet_scale) {
  return run_bwd(bwd_plane_cascade, N, C, H, W, L, K, x, dy, w_base, b_base, w_sub, base_scale,
                 wavelet_scale, dx, dw_base, db_base, dw_sub, dbase_scale, dwavelet_scale);
}

// Form B backward (brute-force transpose and explicit sums; tiny shapes only).
int oracle_bwd_direct(int N, int C, int H, int W, int L, int K, const double* x, const double* dy,
                      const double* w_base, const double* b_base, const double* w_sub,
                      const double* base_scale, const double* wavelet_scale, double* dx, double* dw_base,
                      double* db_base, double* dw_sub, double* dbase_scale, double* dwavelet_scale) {
  return run_bwd(bwd_plane_direct, N, C, H, W, L, K, x, dy, w_base, b_base, w_sub, base_scale,
                 wavelet_scale, dx, dw_base, db_base, dw_sub, dbase_scale, dwavelet_scale);
}

}  // extern "C"
