// Launch plan of the pipelined whole-plane forward / input-gradient kernel
// (fwd2_kernel), shared by the host planner, the kernel and the CPU index
// replay.
//
// A CTA runs two warp groups on a stream of units (P planes of one channel):
//   - the producer group (F2_NF threads) brings the raw planes into shared
//     memory (bulk copies or cp.async, two slots), builds the Haar pyramid
//     (levels 1 and 2 fused over 4x4 blocks, then 3..L), writes the float32
//     input plane in the layout the base convolution reads, convolves the
//     bands of levels 2..L and folds them into one level-1 term R1 by the
//     synthesis cascade;
//   - the consumer group (F2_NB threads) convolves the level-1 bands (Z1) and
//     runs the final strips: base convolution + level-1 synthesis + R1 + bias,
//     stored to HBM.
// The two groups overlap: while the consumers work on unit v, the producers
// already prepare unit v+1.  They hand over through mbarriers (b1ready,
// fready: producer -> consumer; mid: consumer -> producer).
//
// Every convolution is a strip of 4 output columns x F2_SA rows per thread
// (F2_SAC rows for the small coarse levels, which the producer group spreads
// over more threads), read through 16-byte aligned windows; buffer strides
// are chosen by the planner so that consecutive strips fall into consecutive
// 16-byte bank groups (no shared-memory bank conflicts on the window loads).
#pragma once

#include <stdint.h>

#include "wtconv_plan.h"

#define F2_NF 128                 // producer threads (four warps)
#define F2_NB 128                 // consumer threads (four warps)
#define F2_NT (F2_NF + F2_NB)
#define F2_SA 7                   // strip height of the level-1 and final strips: output rows per strip
#define F2_SAC 4                  // strip height of the coarse (levels 2..L) strips
#define F2_NMB 5                  // mbarriers: rawfull[2], b1ready, mid, fready

// A buffer of 4-band (or 1-band) planes: element (p, q) of band b of plane g
// at off + g*plane + b*band + (p + pr)*stride + (q + pc); pr, pc are the
// zero margin before the interior (R for convolution inputs, 0 otherwise).
struct WtF2Buf {
  int off;
  int stride;
  int band;
  int plane;
  int rows;  // allocated rows per band
};

struct WtF2Plan {
  int N, C, H, W, L, K, dtype;
  int P;       // planes per unit
  int G;       // units per channel = ceil(N / P)
  int units;   // C * G
  int Hs[WT_MAXL + 1], Ws[WT_MAXL + 1];
  // Strips per band: level-1 convolutions: A[1] x T[1] strips of F2_SA x 4
  // coefficients; levels l >= 2: A[l] x T[l] strips of F2_SAC x 4; l = 0:
  // the final strips (F2_SA x 4 outputs).
  int A[WT_MAXL + 1], T[WT_MAXL + 1];
  int n1;                         // level-1 convolution strips per plane: 4 * A[1] * T[1]
  int nf;                         // final strips per plane: A[0] * T[0]
  int nco;                        // coarse (levels 2..L) convolution strips per plane
  int co_begin[WT_MAXL + 2];      // first coarse strip of level l within a plane; [L+1] = nco
  int nbh, nbw, na;               // analysis blocks (4x4 input pixels) per plane: rows, cols, total
  // Raw input slots (two): P planes of H*W elements of the activation type,
  // each plane at a 16-byte multiple.
  int raw_off, raw_slot;          // floats
  int raw_pb;                     // bytes per raw plane (16-byte multiple)
  int plane_bytes;                // H * W * element size
  int load_mode;                  // 0: one bulk copy per plane; 1/2/3: cp.async of 16/8/4-byte chunks
  int chunk;                      // bytes per copy chunk (load_mode 1..3)
  WtF2Buf X;                      // float32 input plane: R rows and 4 columns of zero margin; two slots
  int xslot;
  WtF2Buf B[WT_MAXL + 1];         // level-l bands (margin R); B[1] shared, B[2..L] producer-only
  WtF2Buf Z[WT_MAXL + 1];         // convolved bands: Z[1] consumer-only, Z[2..L] producer-only
  WtF2Buf RC[WT_MAXL + 1];        // cascade sums at level m = 1..L-1 (one band); RC[1] = R1, two slots
  int zo;                         // Z1 and R1 column q sits at buffer column q + zo (f2_zo)
  int r1slot;
  int w_off, wb, wslot;           // folded weights: two slots of (1 + 4L) kernels of wb floats
  int mb_off;                     // mbarriers (8-byte aligned), after everything else
  int smem_bytes;
  int out_vec;                    // y rows take 4-element vector stores
  int grid;                       // persistent CTAs
  int wait_shift;                 // bounded waits give up after 2^wait_shift clock cycles
  uint32_t dbg_extra_tx;          // test hook: bytes added to each copy barrier's expected count (0)
  WtDiv d_n1, d_a1t1, d_t1;       // divisions of the level-1 strip index
  WtDiv d_nf, d_tf;               // ... of the final strip index
  WtDiv d_na, d_nbw;              // ... of the analysis block index
  WtDiv d_G;                      // unit -> channel
  WtDiv d_chunks;                 // copy chunks per plane
};

// ---- index helpers shared by the kernel, the planner and the CPU replay ----

#ifdef __CUDACC__
#define F2_HD __host__ __device__ __forceinline__
#else
#define F2_HD inline
#endif

// Float offset of the window (top-left, 16-byte aligned) of level-1
// convolution strip k of a unit, and the strip's coordinates.
struct F2Strip {
  int g, b, r, s;
};

F2_HD F2Strip f2_l1_strip(const WtF2Plan& pl, int k) {
  F2Strip t;
  t.g = wt_fdiv(k, pl.d_n1);
  int rem = k - t.g * pl.n1;
  t.b = wt_fdiv(rem, pl.d_a1t1);
  rem -= t.b * (pl.A[1] * pl.T[1]);
  t.r = wt_fdiv(rem, pl.d_t1);
  t.s = rem - t.r * pl.T[1];
  return t;
}

F2_HD F2Strip f2_final_strip(const WtF2Plan& pl, int k) {
  F2Strip t;
  t.g = wt_fdiv(k, pl.d_nf);
  const int rem = k - t.g * pl.nf;
  t.b = 0;
  t.r = wt_fdiv(rem, pl.d_tf);
  t.s = rem - t.r * pl.T[0];
  return t;
}

// Coarse strip k of a plane (levels 2..L): level, band, strip row, strip column.
F2_HD void f2_coarse_strip(const WtF2Plan& pl, int k, int& l, int& b, int& r, int& s) {
  l = 2;
  while (l < pl.L && k >= pl.co_begin[l + 1]) ++l;
  int rem = k - pl.co_begin[l];
  const int per_band = pl.A[l] * pl.T[l];
  b = rem / per_band;
  rem -= b * per_band;
  r = rem / pl.T[l];
  s = rem - r * pl.T[l];
}

// Window of a convolution strip of sa rows over band b of buffer B (margin
// R on every side): buffer rows sa*r .. sa*r + sa + K - 2, columns from 4s.
F2_HD int f2_win(const WtF2Buf& B, int g, int b, int r, int s, int sa = F2_SA) {
  return B.off + g * B.plane + b * B.band + sa * r * B.stride + 4 * s;
}

// Interior element (p, q) of band b, plane g of a margin-m buffer.
F2_HD int f2_at(const WtF2Buf& B, int g, int b, int p, int q, int m) {
  return B.off + g * B.plane + b * B.band + (p + m) * B.stride + (q + m);
}

// Float32 vector width of a strip window row: ceil((4 + K - 1) / 4) float4s.
F2_HD int f2_nv(int K) { return (K + 6) / 4; }

// Final strips are shifted left by f2_sh(K) = (4 - K/2) mod 4 output columns:
// strip s covers output columns 4s - sh .. 4s - sh + 3.  The input plane X
// keeps a 4-column left margin (its rows are written with aligned 16-byte
// stores), and with the shift the base convolution's window of strip s
// starts at buffer column 4s - sh - K/2 + 4 = 4s: aligned, whatever k.
F2_HD int f2_sh(int K) { return (4 - K / 2) & 3; }
// The level-1 columns of a final strip start at (4s - sh) >> 1 = 2s - sh/2
// (sh even); Z1 and R1 are stored shifted right by f2_zo(K) = sh / 2 columns
// so that this pair starts on an even buffer column (one 8-byte load).
// Odd shifts (k = 3, 7) read single columns.
F2_HD int f2_zo(int K) { return f2_sh(K) == 2 ? 1 : 0; }
