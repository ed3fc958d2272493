// Launch plans shared by the host planner and the kernels of libwtconv.
//
// Every kernel keeps whole (n, c) planes resident in shared memory together
// with their Haar pyramid, so the activations cross HBM exactly once per
// call (technical summary of "Fast and Memory-Efficient Wavelet Convolutions
// via I/O-Aware Reformulation", "Methodology": compute in registers and
// shared memory instead of materialising coefficients in HBM).
#pragma once

#include <stdint.h>

#define WT_MAXL 8  // largest number of decomposition levels

// A shared-memory plane buffer (float32).  The interior element (i, j) of
// band b lives at  off + b*band + (i + pad)*stride + (j + pad).  Everything
// outside the interior (halo, tile-rounding margin) holds zeros.
struct WtBuf {
  int off;     // floats from the start of the plane slot
  int stride;  // floats per row, a multiple of 4
  int pad;     // zero rows/columns before the interior
  int band;    // floats between consecutive bands
};

// Forward / input-gradient pass.  One CTA owns P planes of one channel c
// (n = gi*P .. gi*P+P-1) and runs: load -> Haar analysis levels 1..L ->
// synthesis tiles from level L down to 1 -> store.
struct WtFwdPlan {
  int N, C, H, W, L, K;
  int P;                 // planes per CTA
  int groups;            // ceil(N / P); grid = C * groups
  int Hs[WT_MAXL + 1];   // level sizes, Hs[0] = H, Hs[l] = ceil(Hs[l-1] / 2)
  int Ws[WT_MAXL + 1];
  int tr[WT_MAXL + 1];   // tile rows / columns at level l >= 1 (tiles of TP x TQ)
  int tc[WT_MAXL + 1];
  WtBuf lev[WT_MAXL + 1];  // lev[0] = input plane, lev[l] = 4 coefficient bands of level l
  WtBuf syn[WT_MAXL + 1];  // syn[l] (1 <= l < L): coarse synthesis sum T^l (pad 0, 1 band)
  int plane_floats;      // floats per plane slot
  int w_off;             // folded weights, after the P plane slots
  int w_band;            // floats per folded kernel (k*k rounded up to 4)
  int smem_bytes;
  int vec_ok;            // rows can use 16-byte global accesses (W % elems-per-16B == 0)
};

// Parameter-gradient pass.  One CTA owns channel c and the planes
// n in [gi*chunk, min(N, (gi+1)*chunk)), P at a time.  "Bands" B number the
// correlations: B = 0 base path, B = 1 + 4*(l-1) + b for level l, band b.
struct WtBwPlan {
  int N, C, H, W, L, K;
  int P;                 // planes resident at once
  int chunk;             // planes per CTA
  int groups;            // ceil(N / chunk); grid = C * groups
  int Hs[WT_MAXL + 1];
  int Ws[WT_MAXL + 1];
  int tr[WT_MAXL + 1];   // 4x4-tile rows / columns per level (level 0 = base path)
  int tc[WT_MAXL + 1];
  int item_begin[WT_MAXL + 2];  // first tile item of level l within a plane (l = 0..L), [L+1] = total
  int items_per_plane;
  WtBuf xs[WT_MAXL + 1];  // shifted operand: x (l = 0) and its level-l bands, pad = r
  WtBuf ds[WT_MAXL + 1];  // unshifted operand: dy (l = 0) and its level-l bands, pad = 0
  int plane_floats;
  int smem_bytes;
  int nbands;            // 1 + 4L
  int part_stride;       // floats per (group, channel) partial record = nbands*(k*k+1)
  int vec_ok;
};

#define WT_FWD_THREADS 128
#define WT_BW_THREADS 256
#define WT_BW_MAX_ITEMS 2  // tile items per thread in the parameter-gradient pass
#define WT_TP 2            // forward tile: TP x TQ coefficient positions per level
#define WT_TQ 4
#define WT_BT 4            // parameter-gradient tile: WT_BT x WT_BT positions
