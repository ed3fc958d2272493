// Device functions shared by the whole-plane and the windowed forward /
// input-gradient kernels: weight staging with folded scales and the final
// tiles (base convolution + closed-form synthesis + store).
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805), technical summary, "Methodology":
// scales folded into the weights, synthesis collapsed into one sum indexed
// by the bits of the output coordinate ("Proposition 2").
#pragma once

#include "wtconv_device.cuh"

namespace wt {

// Adds sum_b sign_b(u, v) * z_b to c[u][v] for the four parities (u, v).
__device__ __forceinline__ void add_parities(float z0, float z1, float z2, float z3, float (&c)[2][2]) {
  const float e0 = z0 + z1, e1 = z0 - z1, f0 = z2 + z3, f1 = z2 - z3;
  c[0][0] += e0 + f0;  // (u, v) = (0, 0): all bands +
  c[0][1] += e0 - f0;  // (0, 1): column-high and diagonal -
  c[1][0] += e1 + f1;  // (1, 0): row-high and diagonal -
  c[1][1] += e1 - f1;  // (1, 1): row-high and column-high -
}

// Stages the folded weights of channel c: band 0 = s_base*W_base, band
// 1 + 4(l-1) + b = 4^-l * s_w * W_l,b (all rotated by 180 degrees for the
// input gradient); the padding entries of each band are zero.
template <int K, bool ROT>
__device__ __forceinline__ void stage_weights(float* wsm, int wb, int L, int C, int c,
                                              const float* __restrict__ w_base,
                                              const float* __restrict__ w_sub,
                                              const float* __restrict__ s_base,
                                              const float* __restrict__ s_w, int tid, int nthreads) {
  constexpr int KK = K * K;
  for (int i = tid; i < (1 + 4 * L) * wb; i += nthreads) {
    const int band = i / wb;
    const int t = i - band * wb;
    float v = 0.f;
    if (t < KK) {
      const int ts = ROT ? KK - 1 - t : t;
      if (band == 0) {
        v = s_base[c] * w_base[(size_t)c * KK + ts];
      } else {
        const int l = (band - 1) >> 2, b = (band - 1) & 3;
        const int ch = l * 4 * C + 4 * c + b;
        const float norm = __int_as_float((127 - 2 * (l + 1)) << 23);  // 4^-(l+1), exact
        v = norm * s_w[ch] * w_sub[(size_t)ch * KK + ts];
      }
    }
    wsm[i] = v;
  }
}

// Final tiles of one unit: each thread takes TP x TQ level-1 positions =
// 2TP x 2TQ output pixels (the tile height is a plan choice: TP = 4, or 2
// for small planes), gathers the coarse levels and the level-1 butterflies
// of the synthesis, accumulates the base convolution on top and stores y.
// The tiles cover the plan's final-tile grid (ftr x ftc).  Whole planes:
// xo = gi0 = gj0 = 0 and (Hg, Wg) = (H, W).  Windows: the grid covers the
// output tile, whose first pixel is input-buffer element (xo, xo) and output
// element (gi0, gj0) of an Hg x Wg plane; Z buffers hold the tile's
// coefficients only.  NT threads share the tiles.
template <int K, typename T, int TP, int NT = WT_FWD_THREADS>
__device__ __forceinline__ void final_tiles(const WtFwdPlan& pl, const float* work, const float* xs, const float* wsm,
                                            float bias, T* __restrict__ y, int n0, int c, int np, int tid,
                                            int xo, int gi0, int gj0, int Hg, int Wg) {
  constexpr int R = K / 2;
  constexpr int TQ = WT_TQ;
  const int XF = pl.xf, WF = pl.wf;
  const WtBuf X = pl.lev[0];
  const int L = pl.L, C = pl.C;
  const size_t HW = (size_t)Hg * Wg;
  const int per_plane = pl.ftr * pl.ftc;
  for (int it = tid; it < np * per_plane; it += NT) {
    const int g = fdiv(it, pl.f_pp);
    const int rem = it - g * per_plane;
    const int tp = fdiv(rem, pl.f_c);
    const int p0 = tp * TP, q0 = (rem - tp * pl.ftc) * TQ;
    const float* ps = work + g * WF;
    const float* px = xs + g * XF;

    // Coarse levels 2..L, gathered per level-1 position (p0 + o, q0 + j):
    // level l contributes the parity value (bit l-2 of p, bit l-2 of q) of
    // its coefficients at (p >> (l-1), q >> (l-1)).
    float cc[TP][TQ];
#pragma unroll
    for (int o = 0; o < TP; ++o)
#pragma unroll
      for (int j = 0; j < TQ; ++j) cc[o][j] = bias;
    if (L >= 2) {
      // level 2: rows p0/2 .. p0/2 + TP/2 - 1, column q0/2; parity (o & 1, j)
      const WtBuf Z2 = pl.zb[2];
      const float* z2 = ps + Z2.off + (p0 >> 1) * Z2.stride + (q0 >> 1);
#pragma unroll
      for (int k = 0; k < TP / 2; ++k) {
        const float* zk = z2 + k * Z2.stride;
        float par[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        add_parities(zk[0], zk[Z2.band], zk[2 * Z2.band], zk[3 * Z2.band], par);
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < TQ; ++j) cc[2 * k + u][j] += par[u][j];
      }
    }
    for (int l = 3; l <= L; ++l) {
      // one coarse position per tile; column parity fixed, row parity from bit l-2 of p0 + o
      const WtBuf Zl = pl.zb[l];
      const float* zl = ps + Zl.off + (p0 >> (l - 1)) * Zl.stride + (q0 >> (l - 1));
      float par[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      add_parities(zl[0], zl[Zl.band], zl[2 * Zl.band], zl[3 * Zl.band], par);
      const int v = (q0 >> (l - 2)) & 1;
#pragma unroll
      for (int o = 0; o < TP; ++o) {
        const int u = ((p0 + o) >> (l - 2)) & 1;
        const float add = u ? (v ? par[1][1] : par[1][0]) : (v ? par[0][1] : par[0][0]);
#pragma unroll
        for (int j = 0; j < TQ; ++j) cc[o][j] += add;
      }
    }

    // Level 1 per output parity, plus the coarse sum.
    float out[2 * TP][2 * TQ];
    const WtBuf Z1 = pl.zb[1];
#pragma unroll
    for (int o = 0; o < TP; ++o) {
      const float* z1 = ps + Z1.off + (p0 + o) * Z1.stride + q0;
      float2 zr[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) zr[b] = *reinterpret_cast<const float2*>(z1 + b * Z1.band);
#pragma unroll
      for (int j = 0; j < TQ; ++j) {
        float par[2][2] = {{cc[o][j], cc[o][j]}, {cc[o][j], cc[o][j]}};
        if (j == 0) add_parities(zr[0].x, zr[1].x, zr[2].x, zr[3].x, par);
        else add_parities(zr[0].y, zr[1].y, zr[2].y, zr[3].y, par);
        out[2 * o][2 * j] = par[0][0];
        out[2 * o][2 * j + 1] = par[0][1];
        out[2 * o + 1][2 * j] = par[1][0];
        out[2 * o + 1][2 * j + 1] = par[1][1];
      }
    }

    // Base convolution from the input plane (interior column 0 sits 4 floats
    // into each row, so the window starts 4 - r floats after a 16-byte
    // boundary; xo is a multiple of 4).
    conv_tile_off<K, 2 * TP, 2 * TQ, 4 - R>(px + X.off + (xo + 2 * p0) * X.stride + xo + 2 * q0, X.stride, wsm,
                                            out);

    T* plane = y + ((size_t)(n0 + g) * C + c) * HW;
    const int j0 = gj0 + 2 * q0;
    // One 2TQ-wide store per row: 16 bytes (float32) or 8 bytes (16-bit).
    // Rows start on that boundary when vec_ok (W*sizeof(T) % 16 == 0, base
    // 16-byte aligned) since j0 is a multiple of 2TQ.
    const bool full_row = pl.vec_ok && (j0 + 2 * TQ <= Wg);
#pragma unroll
    for (int oo = 0; oo < 2 * TP; ++oo) {
      const int i = gi0 + 2 * p0 + oo;
      if (i < Hg) {
        T* dst = plane + (size_t)i * Wg + j0;
        if (full_row) {
          stg_row<T, 2 * TQ>(dst, out[oo]);
        } else {
#pragma unroll
          for (int jj = 0; jj < 2 * TQ; ++jj)
            if (j0 + jj < Wg) dst[jj] = from_f32<T>(out[oo][jj]);
        }
      }
    }
  }
}

}  // namespace wt
