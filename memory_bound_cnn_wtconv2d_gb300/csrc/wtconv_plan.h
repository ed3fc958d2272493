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

// Division by a launch-constant divisor d without a hardware divide:
// q = (umulhi(n, mul) + n) >> shift with shift = ceil(log2 d) and
// mul = floor(2^32 (2^shift - d) / d) + 1 (Granlund & Montgomery, "Division
// by invariant integers using multiplication", PLDI 1994).  Exact for
// 0 <= n < 2^24, which bounds every index it is used on.
struct WtDiv {
  uint32_t mul;
  uint32_t shift;
};

// A shared-memory plane buffer (float32).  The interior element (i, j) of
// band b lives at  off + b*band + (i + prow)*stride + (j + pcol).
// Everything outside the interior (halo, tile-rounding margin) holds zeros.
struct WtBuf {
  int off;     // floats from the start of the plane slot
  int stride;  // floats per row, a multiple of 4
  int prow;    // zero rows above the interior
  int pcol;    // zero columns left of the interior
  int band;    // floats between consecutive bands
};

// Forward / input-gradient pass.  A persistent grid walks the C * groups
// units (channel c, planes n = gi*P .. gi*P+P-1) in order; per unit a CTA
// runs: load -> Haar analysis (levels 1 and 2 fused, then 3..L) -> band
// convolutions of every level into Z buffers -> final tiles (base conv +
// bit-indexed synthesis) -> store.
struct WtFwdPlan {
  int N, C, H, W, L, K;
  int P;                 // planes per CTA
  int groups;            // units per channel: ceil(N / P)
  int Hs[WT_MAXL + 1];   // level sizes, Hs[0] = H, Hs[l] = ceil(Hs[l-1] / 2)
  int Ws[WT_MAXL + 1];
  WtBuf lev[WT_MAXL + 1];  // lev[0] = input plane (pcol 4), lev[l] = 4 coefficient bands (pad r)
  WtBuf zb[WT_MAXL + 1];   // zb[l]: the 4 convolved, scale-folded bands of level l (pad 0)
  int ztr[WT_MAXL + 1];    // band-convolution tiles (WT_ZT x WT_ZT) per level: rows, columns
  int ztc[WT_MAXL + 1];
  int zbegin[WT_MAXL + 2];  // first (band, tile) item of level l within a plane; [L+1] = total
  int zipp;                 // band-convolution items per plane
  int ftp;                  // level-1 rows per final tile: WT_TP, or WT_TP / 2 for small planes
  int ftr, ftc;             // final tiles (ftp x WT_TQ level-1 positions) per plane: rows, columns
  int xf;                // floats per input-plane buffer (= TMA box of one plane)
  int xslot;             // floats per input buffer set (P planes, 128-byte multiple)
  int nsets;             // input sets: 2 (the next unit streams in meanwhile) or 1
  int stage_off;         // = xslot: second set, or (16-bit) the staging area of the raw planes
  int wf;                // floats per work area (pyramid + convolved bands; P of them)
  int work_off;          // after the input sets / staging area
  int w_off;             // folded weights, after the work areas
  int w_band;            // floats per folded kernel (k*k rounded up to 4)
  int mb_off;            // two mbarriers (8-byte aligned), after the weights
  int smem_bytes;
  int vec_ok;            // rows can use 16-byte global accesses (W % elems-per-16B == 0)
  int use_tma;           // input planes arrive by TMA box copies (float32, 16-byte rows)
  uint32_t tma_bytes;    // bytes of one box (P planes)
  int use_bulk;          // 16-bit planes are staged raw, then widened: 1 = bulk copies, 2 = 8-byte cp.async
  uint32_t bulk_bytes;   // bytes of one raw 16-bit plane (H*W*2: a multiple of 16, or of 8 for cp.async)
  WtDiv cp_pp;           // 8-byte chunks per raw plane (H*W/4), for the cp.async staging
  int wd_vec;            // elements per widening item: 4 (W % 4 == 0), 2 (W even) or 1
  WtDiv wd_pp, wd_w;     // widening: items per plane, items per row
  WtDiv ld_pp, ld_w;     // plane load: items per plane, items per row
  WtDiv an_pp[WT_MAXL + 1], an_w[WT_MAXL + 1];  // analysis at level l (l = 2: the fused 1+2 pass)
  WtDiv z_ipp;                                  // band-convolution items per plane
  WtDiv z_tiles[WT_MAXL + 1], z_tc[WT_MAXL + 1];  // ztr*ztc and ztc per level
  WtDiv f_pp, f_c;                              // final tiles per plane, per row
  // Windowed mode, for planes whose pyramid does not fit one CTA: a unit is
  // one th x tw output tile of P planes of one channel.  The CTA loads the
  // tile's window, the tile plus `halo` pixels on every side (zero outside
  // the H x W plane), builds the Haar pyramid of the whole window, and
  // convolves the bands and runs the final tiles on the tile only.  Hs/Ws and
  // lev[] then describe the window (Hs[0] x Ws[0] pixels), ztr/ztc, zb[] and
  // ftr/ftc the tile; H and W stay the plane's.
  int win;               // 1 = windowed mode
  int halo;              // h: 2^L * r rounded up to 8 (a multiple of 2^L, and of 8 for 16-byte rows)
  int th, tw;            // output tile, multiples of max(2^L, 8)
  int nty, ntx;          // tiles per plane
  int zo[WT_MAXL + 1];   // h >> l: the tile's first level-l coefficient row / column in the window
  int win_load;          // 0 = plain loads, 1 = float32 box copy (margins included), 2 = 16-bit box copy into
                         // the staging area, widened per unit
  // Bounded waits on the plane copies give up after 2^wait_shift clock
  // cycles; each copy barrier expects dbg_extra_tx bytes more than its copies
  // deliver.  31 and 0 in normal operation (set at launch; the test hook
  // wtconv_test_copy_timeout shortens the limit and arms the extra bytes so
  // that every wait runs out).
  int wait_shift;
  uint32_t dbg_extra_tx;
};

// Parameter-gradient pass.  The work is C * batches units (channel c, batch
// of P planes), split evenly and in order over a persistent grid; a CTA
// correlates one unit at a time (the next unit's planes stream in meanwhile
// when there are two input sets) and writes one record per channel it
// touched.  "Bands" B number the correlations: B = 0 base path,
// B = 1 + 4*(l-1) + b for level l, band b.
struct WtBwPlan {
  int N, C, H, W, L, K;
  int P;                 // planes per unit
  int batches;           // units per channel = ceil(N / P)
  WtDiv nb_div;          // divides by batches
  int grid;              // persistent CTAs G; CTA i starts at unit floor(U*i/G) = uq*i + (ur*i)/G
  int uq, ur;            // U = C * batches = uq*G + ur
  WtDiv g_div;           // divides by G (exact: ur*i < G^2 < 2^24)
  int nrec;              // record slots per CTA (most channels one CTA touches)
  int Hs[WT_MAXL + 1];
  int Ws[WT_MAXL + 1];
  int tbr;               // tile rows: 8 (one tile per thread) or 4 (up to two per thread)
  int mi;                // tiles per thread: 1, or 2 (4-row tiles of the whole-plane gradient pass)
  int tcw;               // tile columns: 4
  int tr[WT_MAXL + 1];   // tbr x tcw tiles per level (level 0 = base path): rows, columns
  int tc[WT_MAXL + 1];
  int item_begin[WT_MAXL + 2];  // first tile item of level l within a plane (l = 0..L), [L+1] = total
  int items_per_plane;
  WtBuf xs[WT_MAXL + 1];  // shifted operand: x (l = 0: r zero rows, 4 zero columns) and its level-l bands, pad r
                          // (whole-plane plans: r zero rows and a right margin only, which is the next row's left one)
  WtBuf ds[WT_MAXL + 1];  // unshifted operand: dy (l = 0, pad 0) and its level-l bands, pad 0
  int xbf, dbf;          // floats per raw x plane / raw dy plane (= one TMA box row set of one plane)
  int xr;                // offset of the dy planes within an input set (128-byte multiple)
  int islot;             // floats per input set (P x planes, then P dy planes)
  int nsets;             // input sets: 2 (the next batch streams in meanwhile) or 1
  int wf;                // floats per work area (both pyramids; P of them)
  int work_off;          // = nsets * islot
  int red_floats;        // work area = max(P work areas, end-of-channel reduction), floats
  int mb_off;            // two mbarriers (8-byte aligned), after everything else
  int smem_bytes;
  int use_tma;           // input planes arrive by TMA box copies (float32, 16-byte rows)
  uint32_t tma_bytes;    // bytes of one input set (x and dy boxes)
  int stage_off;         // 16-bit staging area (raw x planes, then raw dy planes), floats; 0 = none
  int use_bulk;          // 16-bit planes are staged raw, then widened: 1 = bulk copies, 2 = 8-byte cp.async
  uint32_t bulk_bytes;   // bytes of one raw 16-bit plane (H*W*2: a multiple of 16, or of 8 for cp.async)
  WtDiv cp_pp;           // 8-byte chunks per raw plane (H*W/4), for the cp.async staging
  int wd_vec;            // elements per widening item: 4 (W % 4 == 0), 2 (W even) or 1
  WtDiv wd_pp, wd_w;     // widening: items per plane, items per row
  int nbands;            // 1 + 4L
  int part_stride;       // floats per (group, channel) partial record = nbands*(k*k+1)
  int vec_ok;
  WtDiv ld_pp, ld_w;
  WtDiv an_pp[WT_MAXL + 1], an_w[WT_MAXL + 1];
  WtDiv ipp;                                   // items per plane
  WtDiv tiles[WT_MAXL + 1], tcd[WT_MAXL + 1];  // tr*tc and tc per level
  // Windowed mode, for planes beyond one CTA: a unit is one th x tw tile of
  // P planes of one channel, and `batches` counts the units of a channel
  // (plane groups x tiles).  x arrives as the tile's window (the tile plus
  // `halo` pixels on every side, zero outside the plane) and dy as the tile
  // alone: tiles start at multiples of 2^L, so the tile's dy coefficients
  // depend on the tile only.  Hs/Ws and xs[] then describe the x window,
  // dHs/dWs and ds[] the dy tile, tr/tc the correlation tiles over the tile.
  int win;               // 1 = windowed mode
  int halo;              // h: 2^L * r rounded up to 8
  int th, tw;            // tile, multiples of max(2^L, 8)
  int nty, ntx;          // tiles per plane
  int groups;            // plane groups per channel: ceil(N / P)
  int dHs[WT_MAXL + 1], dWs[WT_MAXL + 1];  // dy tile pyramid: th >> l, tw >> l
  int zo[WT_MAXL + 1];   // h >> l: the tile's first level-l coefficient in the x window
  int win_load;          // 0 = plain loads, 1 = float32 box copies, 2 = 16-bit box copies into the staging area
  WtDiv dn_pp[WT_MAXL + 1], dn_w[WT_MAXL + 1];  // analysis of the dy tile (l = 2: the fused 1+2 pass)
  WtDiv dld_pp, dld_w;   // plain loads of the dy tile: items per tile, per row
  WtDiv dwd_pp, dwd_w;   // widening of the raw 16-bit dy tiles: items per tile, per row
  int stage_dx;          // 16-bit staging: floats from the staging area's start to the raw dy tiles
  int wait_shift;        // as in WtFwdPlan
  uint32_t dbg_extra_tx;
};

#define WT_SMEM_SLACK 128  // bytes added to every dynamic shared-memory size for 128-byte realignment
#define WT_FWD_THREADS 128
#define WT_BW_THREADS 256
#define WT_BW_MAX_ITEMS 2  // tile items per thread in the parameter-gradient pass
#define WT_TP 4            // final tile: TP x TQ level-1 positions = 2TP x 2TQ outputs
#define WT_TQ 2
#define WT_ZT 4            // band-convolution tile: ZT x ZT coefficient positions
#define WT_BT 4            // parameter-gradient tile: WT_BT x WT_BT positions

// Division helpers shared by the host planner and the kernels.
#ifdef __CUDACC__
#define WT_HD __host__ __device__ __forceinline__
#else
#define WT_HD inline
#endif
WT_HD int wt_fdiv(int n, WtDiv d) {
  return (int)(((uint32_t)(((uint64_t)(uint32_t)n * d.mul) >> 32) + (uint32_t)n) >> d.shift);
}
// First (channel, batch) unit of persistent CTA i: floor(U*i/G).
WT_HD int bw_unit_begin(const WtBwPlan& pl, int i) { return pl.uq * i + wt_fdiv(pl.ur * i, pl.g_div); }
