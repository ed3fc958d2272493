// WTConv2d parameter gradients (sm_103a).
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805); the technical summary's "Key
// contributions" state that the fused implementation reproduces all
// parameter gradients.  With the scales folded into the weights
// (summary, "Methodology", folding learned scales), every parameter
// gradient follows from raw correlation sums:
//
//   base:     G_0[t]   = sum_{n,i,j} dy[i][j] * x[i+du-r][j+dv-r],   g = sum dy
//   level l:  G_lb[t]  = sum_{n,p,q} D^l_b[p][q] * Y^l_b[p+du-r][q+dv-r]
//
// where Y^l = F_l x and D^l = F_l dy are the level-l Haar coefficients of x
// and of dy (dL/dZ^l = F_l dy because the synthesis is F_l^T), and then
//   dW_base = s_b G_0, db = s_b g, ds_b = <W_base, G_0> + b g,
//   dW_l = s_w G_l,    ds_w = <W_l, G_l>.
//
// A persistent grid splits the (channel, batch-of-planes) units evenly and in
// order.  Planes of x and dy are read once into shared memory, both pyramids
// are rebuilt there (unnormalised, so G_l is recovered as 4^-l times the
// sum), and every thread accumulates the K*K correlations of its fixed tiles
// in registers across the units of one channel.  When a CTA leaves a channel
// the tile sums of each band are reduced through shared memory into one
// record per (CTA, channel); a second kernel adds the records of each channel
// in CTA order, so the result does not depend on scheduling.
#include "wtconv_device.cuh"
#include "wtconv_launch.h"

#include <mutex>

namespace wt {

// Bounded waits that gave up (see mbar_wait_bounded); read by take_bw_faults().
static __device__ unsigned int g_bw_faults;

// TR = 8: 8x4 tiles, one per thread; TR = 4: 4x4 tiles, MI (one or two) per
// thread.  Tiles are 4 columns wide so neighbouring lanes read neighbouring
// 16-byte chunks of a row (no shared-memory bank conflicts within a row).
// 16-bit instances are held to the registers of three CTAs per SM with one
// tile per thread at k <= 5 (two at k = 7), and of two CTAs with two tiles
// at k <= 5; the float32 ones are left to the compiler (0: no minimum),
// which fits those by itself.
template <int K, typename T, int TR, int MI>
__global__ void __launch_bounds__(WT_BW_THREADS,
                                  sizeof(T) == 4 ? 0 : K <= 5 ? (MI == 1 ? 3 : 2) : (K == 7 && MI == 1 ? 2 : 0))
    bw_kernel(const __grid_constant__ WtBwPlan pl, const __grid_constant__ CUtensorMap tmx,
              const __grid_constant__ CUtensorMap tmd, const T* __restrict__ x, const T* __restrict__ dy,
              float* __restrict__ part) {
  extern __shared__ __align__(16) float sm_raw[];
  float* const sm = align_smem128(sm_raw);  // TMA box destinations need 128-byte alignment
  constexpr int KK = K * K;
  constexpr int NT = WT_BW_THREADS;
  static_assert(MI == 1 || (TR == 4 && MI == WT_BW_MAX_ITEMS), "two items per thread with 4-row tiles only");
  constexpr int TC = 4;
  constexpr bool ASYNC = sizeof(T) == 4;
  constexpr int R = K / 2;
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L, P = pl.P, NB = pl.batches;
  // Persistent CTA: an even share of the C * NB (channel, batch) units, in
  // order, so it touches one or a few consecutive channels.
  const int u_begin = bw_unit_begin(pl, blockIdx.x);
  const int u_end = bw_unit_begin(pl, blockIdx.x + 1);
  const int c_first = fdiv(u_begin, pl.nb_div);
  const int XBF = pl.xbf, DBF = pl.dbf, WF = pl.wf;
  const int ipp = pl.items_per_plane;
  float* const work = sm + pl.work_off;
  const float* const xf = reinterpret_cast<const float*>(x);
  const float* const dyf = reinterpret_cast<const float*>(dy);
  // TMA path (float32, 16-byte rows): one thread issues the x and dy box
  // copies of a unit into input set `s`; both complete on mbar[s].
  const bool tma = ASYNC && pl.use_tma;
  const bool dbl = pl.nsets == 2;
  uint64_t* const mbar = reinterpret_cast<uint64_t*>(sm + pl.mb_off);
  __shared__ int s_ok;
  uint32_t parity = 0;  // thread 0: phase parity of mbar[0] (bit 0) and mbar[1] (bit 1)
  auto unit_c = [&](int u) { return fdiv(u, pl.nb_div); };
  auto issue = [&](int u, int s) {
    const int cc = unit_c(u);
    const int n0 = (u - cc * NB) * P;
    float* const dst = sm + s * pl.islot;
    fence_proxy_async();  // earlier generic accesses of the set precede the copies
    mbar_arrive_expect_tx(&mbar[s], pl.tma_bytes + pl.dbg_extra_tx);
    tma_load_4d(dst, &tmx, -4, -R, cc, n0, &mbar[s]);
    tma_load_4d(dst + pl.xr, &tmd, 0, 0, cc, n0, &mbar[s]);
  };
  auto prefetch = [&](int u) {  // the boxes issue(u, .) will copy, into L2
    const int cc = unit_c(u);
    const int n0 = (u - cc * NB) * P;
    tma_prefetch_4d(&tmx, -4, -R, cc, n0);
    tma_prefetch_4d(&tmd, 0, 0, cc, n0);
  };
  // 16-bit staged path: a unit's raw x and dy planes land in the staging area
  // (one bulk copy per plane on mbar[0], or 8-byte cp.async chunks from every
  // thread); the unit widens them into its input set, after which the next
  // unit's copies are issued.
  const bool bulk = !ASYNC && pl.use_bulk == 1;
  const bool cpa = !ASYNC && pl.use_bulk == 2;  // same staging, filled by every thread's 8-byte cp.async
  const bool staged = bulk || cpa;
  const int HWp = pl.H * pl.W;
  T* const stage_x = reinterpret_cast<T*>(sm + pl.stage_off);
  T* const stage_d = stage_x + P * HWp;
  auto issue_bulk = [&](int u) {
    const int cc = unit_c(u);
    const int n0 = (u - cc * NB) * P;
    const int npp = min(P, pl.N - n0);
    fence_proxy_async();  // the widening reads of the staging area precede the copies
    mbar_arrive_expect_tx(&mbar[0], 2u * (uint32_t)npp * pl.bulk_bytes + pl.dbg_extra_tx);
    for (int g = 0; g < npp; ++g) {
      const size_t src = ((size_t)(n0 + g) * C + cc) * HWp;
      bulk_load(stage_x + g * HWp, x + src, pl.bulk_bytes, &mbar[0]);
      bulk_load(stage_d + g * HWp, dy + src, pl.bulk_bytes, &mbar[0]);
    }
  };
  auto issue_cpa = [&](int u) {
    const int cc = unit_c(u);
    const int n0 = (u - cc * NB) * P;
    const int chunks = HWp >> 2;  // 8-byte chunks (4 elements) per plane
    const int total = min(P, pl.N - n0) * chunks;
    for (int i = tid; i < total; i += NT) {
      const int g = fdiv(i, pl.cp_pp);
      const int o = (i - g * chunks) << 2;
      const size_t src = ((size_t)(n0 + g) * C + cc) * HWp + o;
      cp_async8(reinterpret_cast<float*>(stage_x + g * HWp + o), reinterpret_cast<const float*>(x + src));
      cp_async8(reinterpret_cast<float*>(stage_d + g * HWp + o), reinterpret_cast<const float*>(dy + src));
    }
    cp_async_commit();
  };
  auto load_async = [&](int u, int s) {
    const int cc = unit_c(u);
    const int n0 = (u - cc * NB) * P;
    const int np = min(P, pl.N - n0);
    float* const dst = sm + s * pl.islot;
    load_planes_async(dst, XBF, pl.xs[0], xf, n0, np, cc, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
    load_planes_async(dst + pl.xr, DBF, pl.ds[0], dyf, n0, np, cc, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w,
                      tid, NT);
    cp_async_commit();
  };

  // Zeroed once: interiors are rewritten per unit, margins stay zero (the box
  // copies write whole padded planes themselves).  The work area is zeroed
  // again after each channel's reduction, which reuses it.
  if (tma) zero_smem(work, pl.red_floats, tid, NT);
  else zero_smem(sm, pl.work_off + pl.red_floats, tid, NT);

  float acc[MI][KK];
  float gs[MI];
#pragma unroll
  for (int s = 0; s < MI; ++s) {
    gs[s] = 0.f;
#pragma unroll
    for (int t = 0; t < KK; ++t) acc[s][t] = 0.f;
  }
  if ((tma || bulk) && tid == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (tma) {
    if (tid == 0 && u_begin < u_end) issue(u_begin, 0);
  } else if (bulk) {
    if (tid == 0 && u_begin < u_end) issue_bulk(u_begin);
  } else if (cpa) {
    if (u_begin < u_end) issue_cpa(u_begin);
  } else if (ASYNC && dbl && u_begin < u_end) {  // first unit
    load_async(u_begin, 0);
    cp_async_wait_all();
  }
  int slot = 0;
  for (int u = u_begin; u < u_end;) {
    // The units of channel c held by this CTA: [u, u_stop).
    const int c = unit_c(u);
    const int u_stop = min(u_end, (c + 1) * NB);
    for (; u < u_stop; ++u, slot = dbl ? slot ^ 1 : 0) {
      const int n0 = (u - c * NB) * P;
      const int np = min(P, pl.N - n0);
      float* const in_x = sm + slot * pl.islot;  // this unit's raw x planes
      float* const in_d = in_x + pl.xr;          // ... and raw dy planes
      if (tma) {
        if (tid == 0) {
          const bool ok = mbar_wait_bounded(&mbar[slot], (parity >> slot) & 1u, pl.wait_shift);
          parity ^= 1u << slot;
          if (ok && dbl && u + 1 < u_end) issue(u + 1, slot ^ 1);  // the other set was last read by unit u-1
          if (ok && !dbl && u + 1 < u_end) prefetch(u + 1);       // single set: the copy comes later, from L2
          s_ok = ok;
        }
      } else if (bulk) {
        if (tid == 0) {
          s_ok = mbar_wait_bounded(&mbar[0], parity & 1u, pl.wait_shift);
          parity ^= 1u;
        }
      } else if (cpa) {
        cp_async_wait_all();  // this thread's copies of unit u; the barrier below publishes all
      } else if (!ASYNC || !dbl) {
        load_planes<T>(in_x, XBF, pl.xs[0], x, n0, np, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
        load_planes<T>(in_d, DBF, pl.ds[0], dy, n0, np, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
      } else if (u + 1 < u_end) {  // prefetch the next unit into the other set
        load_async(u + 1, slot ^ 1);
      }
      __syncthreads();  // this unit's planes are visible
      if ((tma || bulk) && !s_ok) {  // the copy did not complete in time: record it and stop (uniform exit)
        const int mb = bulk ? 0 : slot;
        if (tid == 0) {
          atomicAdd(&g_bw_faults, 1u);
          mbar_wait_bounded(&mbar[mb], ((parity >> mb) & 1u) ^ 1u, pl.wait_shift);  // let the copy in flight land
        }
        __syncthreads();
        return;  // records are not written: the caller sees the fault count
      }
      // 16-bit raw planes: widened by the fused level-1/2 pass itself where
      // rows are whole 4-element groups, else first, by a pass of their own.
      // The next unit's copies follow once they are consumed.
      const bool widen12 = staged && L >= 2 && (pl.W & 3) == 0;
      if (staged && !widen12) {
        widen_planes<T>(in_x, XBF, pl.xs[0], stage_x, np, pl.H, pl.W, pl.wd_vec, pl.wd_pp, pl.wd_w, tid, NT);
        widen_planes<T>(in_d, DBF, pl.ds[0], stage_d, np, pl.H, pl.W, pl.wd_vec, pl.wd_pp, pl.wd_w, tid, NT);
        __syncthreads();
        if (bulk && tid == 0 && u + 1 < u_end) issue_bulk(u + 1);
        if (cpa && u + 1 < u_end) issue_cpa(u + 1);
      }

      // Both pyramids: levels 1+2 fused, then 3..L.
      if (L == 1) {
        haar_level(in_x, XBF, work, WF, np, pl.xs[0], pl.xs[1], pl.Hs[1], pl.Ws[1], pl.an_pp[1], pl.an_w[1], tid, NT);
        haar_level(in_d, DBF, work, WF, np, pl.ds[0], pl.ds[1], pl.Hs[1], pl.Ws[1], pl.an_pp[1], pl.an_w[1], tid, NT);
      } else if (widen12) {
        if constexpr (!ASYNC)  // (16-bit instances only)
          widen_levels12_pair<T>(stage_x, in_x, XBF, pl.xs[0], pl.xs[1], pl.xs[2], stage_d, in_d, DBF, pl.ds[0],
                                 pl.ds[1], pl.ds[2], pl.H, pl.W, work, WF, np, pl.Hs[1], pl.Ws[1], pl.Hs[2],
                                 pl.Ws[2], pl.an_pp[2], pl.an_w[2], tid, NT);
      } else {
        haar_levels12_pair(in_x, XBF, pl.xs[0], pl.xs[1], pl.xs[2], in_d, DBF, pl.ds[0], pl.ds[1], pl.ds[2], work,
                           WF, np, pl.Hs[1], pl.Ws[1], pl.Hs[2], pl.Ws[2], pl.an_pp[2], pl.an_w[2], tid, NT);
      }
      __syncthreads();
      if (widen12) {  // the raw planes are consumed: start the next unit's copies
        if (bulk && tid == 0 && u + 1 < u_end) issue_bulk(u + 1);
        if (cpa && u + 1 < u_end) issue_cpa(u + 1);
      }
      for (int l = 3; l <= L; ++l) {
        haar_level_pair(work, WF, work, WF, np, pl.xs[l - 1], pl.xs[l], pl.ds[l - 1], pl.ds[l], pl.Hs[l], pl.Ws[l],
                        pl.an_pp[l], pl.an_w[l], tid, NT);
        __syncthreads();
      }
#pragma unroll
      for (int s = 0; s < MI; ++s) {
        const int item = tid + s * NT;
        if (item < P * ipp) {
          const int g = fdiv(item, pl.ipp);
          if (g < np) {
            const int local = item - g * ipp;
            int l = 0;
            while (l < L && local >= pl.item_begin[l + 1]) ++l;
            const int tiles = pl.tr[l] * pl.tc[l];
            const int rel = local - pl.item_begin[l];
            const int b = fdiv(rel, pl.tiles[l]);
            const int t = rel - b * tiles;
            const int tp = fdiv(t, pl.tcd[l]);
            const int p0 = tp * TR, q0 = (t - tp * pl.tc[l]) * TC;
            const WtBuf Xb = pl.xs[l], Db = pl.ds[l];
            if (l > 0 && pl.Hs[l] <= 2 && pl.Ws[l] <= 2) {  // the whole band (at most 16 products)
              const float* ps = work + g * WF;
              tiny_band_corr<K>(ps + Xb.off + b * Xb.band + Xb.prow * Xb.stride + Xb.pcol, Xb.stride,
                                ps + Db.off + b * Db.band + Db.prow * Db.stride + Db.pcol, Db.stride, acc[s]);
            } else {
              // One instance for every level: x's interior starts pcol floats
              // into a row (4 for the raw plane, 0 for the bands, whose left
              // margin is the previous row's right one), so the window starts
              // 4 - r floats after a 16-byte boundary; dy has no margins.
              const float* xb = l == 0 ? in_x + g * XBF : work + g * WF + b * Xb.band;
              const float* db = l == 0 ? in_d + g * DBF : work + g * WF + b * Db.band;
              const float sum = corr_tile<K, TR, TC, 4 - R>(xb + Xb.off + p0 * Xb.stride + q0 + Xb.pcol - 4, Xb.stride,
                                                            db + Db.off + p0 * Db.stride + q0, Db.stride, acc[s]);
              if (l == 0) gs[s] += sum;
            }
          }
        }
      }
      if (ASYNC && !tma && dbl) cp_async_wait_all();  // this thread's copies of the next unit have landed
      __syncthreads();                                // ... and every read of this unit is done

      if (tma && !dbl && tid == 0 && u + 1 < u_end) issue(u + 1, 0);  // single set: refill it now
    }
    // Leaving channel c: tile sums -> shared memory (the work area) -> one
    // record per band -> this CTA's record slot for c.
    float* const red = work;
    const int rs = KK + 1;
#pragma unroll
    for (int s = 0; s < MI; ++s) {
      const int item = tid + s * NT;
      if (item < P * ipp) {
#pragma unroll
        for (int t = 0; t < KK; ++t) red[item * rs + t] = acc[s][t];
        red[item * rs + KK] = gs[s];
      }
      gs[s] = 0.f;
#pragma unroll
      for (int t = 0; t < KK; ++t) acc[s][t] = 0.f;
    }
    __syncthreads();
    float* rec = part + ((size_t)blockIdx.x * pl.nrec + (c - c_first)) * pl.part_stride;
    for (int qd = tid; qd < pl.nbands * rs; qd += NT) {
      const int B = qd / rs;
      const int t = qd - B * rs;
      const int l = (B == 0) ? 0 : 1 + ((B - 1) >> 2);
      const int b = (B == 0) ? 0 : ((B - 1) & 3);
      const int tiles = pl.tr[l] * pl.tc[l];
      const int first = pl.item_begin[l] + b * tiles;
      float sum = 0.f;
      if (B == 0 || t < KK) {
        for (int g = 0; g < P; ++g)
          for (int i = 0; i < tiles; ++i) sum += red[(g * ipp + first + i) * rs + t];
      }
      rec[qd] = sum;
    }
    __syncthreads();
    if (u < u_end) {
      zero_smem(work, pl.red_floats, tid, NT);  // restore the pyramids' zero margins
      __syncthreads();
    }
  }
}

// Adds the records of channel c from every CTA whose units cover it, in CTA
// order, and unfolds the scales.  One warp per (channel, band): lane t owns
// taps t, t+32, t+64; the scale gradient <W, G> is reduced with a fixed
// shuffle tree, so the result does not depend on scheduling.
__global__ void bw_finalize_kernel(const __grid_constant__ WtBwPlan pl, const float* __restrict__ part,
                                   const float* __restrict__ w_base, const float* __restrict__ b_base,
                                   const float* __restrict__ w_sub, const float* __restrict__ s_base,
                                   const float* __restrict__ s_w, float* __restrict__ dw_base,
                                   float* __restrict__ db_base, float* __restrict__ dw_sub,
                                   float* __restrict__ ds_base, float* __restrict__ ds_w) {
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int C = pl.C, K = pl.K, KK = K * K, rs = KK + 1, NB = pl.batches, G = pl.grid;
  if (warp >= C * pl.nbands) return;  // whole warps exit together
  const int c = warp / pl.nbands;
  const int B = warp - c * pl.nbands;
  // CTAs i0 .. i1-1 hold the units [c*NB, (c+1)*NB) of channel c: i0 holds
  // unit c*NB, i1 is the first CTA starting at or after (c+1)*NB.
  int i0 = (int)((long long)c * G / C);
  while (i0 > 0 && bw_unit_begin(pl, i0) > c * NB) --i0;
  while (bw_unit_begin(pl, i0 + 1) <= c * NB) ++i0;
  int i1 = (int)((long long)(c + 1) * G / C);
  if (i1 < i0 + 1) i1 = i0 + 1;
  while (i1 > i0 + 1 && bw_unit_begin(pl, i1 - 1) >= (c + 1) * NB) --i1;
  while (i1 < G && bw_unit_begin(pl, i1) < (c + 1) * NB) ++i1;
  int l = 0;
  size_t ch = 0;
  float scale;
  const float* w;
  float* dw;
  if (B == 0) {
    scale = s_base[c];
    w = w_base + (size_t)c * KK;
    dw = dw_base + (size_t)c * KK;
  } else {
    l = 1 + ((B - 1) >> 2);
    ch = (size_t)(l - 1) * 4 * C + 4 * c + ((B - 1) & 3);
    scale = s_w[ch];
    w = w_sub + ch * KK;
    dw = dw_sub + ch * KK;
  }
  // Sum the records in CTA order; lane j of each 32-CTA batch finds the
  // record of CTA base + j, the others read it through a shuffle.
  float Gt[3] = {0.f, 0.f, 0.f};  // taps lane, lane + 32, lane + 64 (k <= 9)
  float gsum = 0.f;
  for (int base = i0; base < i1; base += 32) {
    const int i = base + lane;
    long long off = 0;
    if (i < i1) off = ((long long)i * pl.nrec + (c - fdiv(bw_unit_begin(pl, i), pl.nb_div))) * pl.part_stride + (long long)B * rs;
    const int n = min(32, i1 - base);
    for (int j = 0; j < n; ++j) {
      const float* rec = part + __shfl_sync(0xffffffffu, off, j);
#pragma unroll
      for (int m = 0; m < 3; ++m)
        if (lane + 32 * m < KK) Gt[m] += rec[lane + 32 * m];
      if (B == 0 && lane == 0) gsum += rec[KK];
    }
  }
  float dot = 0.f;
#pragma unroll
  for (int m = 0; m < 3; ++m) {
    const int t = lane + 32 * m;
    if (t < KK) {
      const float Gs = ldexpf(Gt[m], -2 * l);  // level-l sums were taken on unnormalised coefficients
      dw[t] = scale * Gs;
      dot = fmaf(w[t], Gs, dot);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (lane == 0) {
    if (B == 0) {
      if (db_base) db_base[c] = scale * gsum;
      ds_base[c] = b_base ? fmaf(b_base[c], gsum, dot) : dot;
    } else {
      ds_w[ch] = dot;
    }
  }
}

template <int K, typename T>
static cudaError_t launch_bw_t(const WtBwPlan& pl, const CUtensorMap& tmx, const CUtensorMap& tmd, const void* x,
                               const void* dy, float* part, cudaStream_t stream) {
  auto kern = pl.tbr == 8   ? bw_kernel<K, T, 8, 1>
              : pl.mi == 1 ? bw_kernel<K, T, 4, 1>
                           : bw_kernel<K, T, 4, WT_BW_MAX_ITEMS>;
  cudaError_t e = ensure_smem((const void*)kern, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)pl.grid;
  kern<<<grid, WT_BW_THREADS, pl.smem_bytes, stream>>>(pl, tmx, tmd, static_cast<const T*>(x),
                                                       static_cast<const T*>(dy), part);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_bw_k(const WtBwPlan& pl, const CUtensorMap& tmx, const CUtensorMap& tmd, const void* x,
                               const void* dy, float* part, cudaStream_t stream) {
  switch (pl.K) {
    case 3: return launch_bw_t<3, T>(pl, tmx, tmd, x, dy, part, stream);
    case 5: return launch_bw_t<5, T>(pl, tmx, tmd, x, dy, part, stream);
    case 7: return launch_bw_t<7, T>(pl, tmx, tmd, x, dy, part, stream);
    case 9: return launch_bw_t<9, T>(pl, tmx, tmd, x, dy, part, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_weight(const WtBwPlan& pl, const CUtensorMap& tmx, const CUtensorMap& tmd, int dtype,
                              const void* x, const void* dy,
                              const float* w_base, const float* b_base, const float* w_sub,
                              const float* s_base, const float* s_w, float* dw_base, float* db_base,
                              float* dw_sub, float* ds_base, float* ds_w, float* part,
                              cudaStream_t stream) {
  cudaError_t e;
  if (dtype == 0) e = launch_bw_k<float>(pl, tmx, tmd, x, dy, part, stream);
  else if (dtype == 1) e = launch_bw_k<__half>(pl, tmx, tmd, x, dy, part, stream);
  else e = launch_bw_k<__nv_bfloat16>(pl, tmx, tmd, x, dy, part, stream);
  if (e != cudaSuccess) return e;
  return launch_bw_finalize(pl, part, w_base, b_base, w_sub, s_base, s_w, dw_base, db_base, dw_sub, ds_base, ds_w,
                            stream);
}

cudaError_t launch_bw_finalize(const WtBwPlan& pl, const float* part, const float* w_base, const float* b_base,
                               const float* w_sub, const float* s_base, const float* s_w, float* dw_base,
                               float* db_base, float* dw_sub, float* ds_base, float* ds_w, cudaStream_t stream) {
  const int warps = pl.C * pl.nbands;
  const int threads = 256;
  bw_finalize_kernel<<<(warps * 32 + threads - 1) / threads, threads, 0, stream>>>(
      pl, part, w_base, b_base, w_sub, s_base, s_w, dw_base, db_base, dw_sub, ds_base, ds_w);
  return cudaGetLastError();
}

// The kernel instance a plan launches (nullptr for an unsupported k).
static const void* bw_pick(const WtBwPlan& pl, int dtype) {
  const void* f = nullptr;
#define WT_BW_PICK(KK, TT)                                         \
  f = pl.tbr == 8   ? (const void*)bw_kernel<KK, TT, 8, 1>         \
      : pl.mi == 1 ? (const void*)bw_kernel<KK, TT, 4, 1>          \
                   : (const void*)bw_kernel<KK, TT, 4, WT_BW_MAX_ITEMS>
#define WT_BW_PICK_K(TT)              \
  switch (pl.K) {                     \
    case 3: WT_BW_PICK(3, TT); break; \
    case 5: WT_BW_PICK(5, TT); break; \
    case 7: WT_BW_PICK(7, TT); break; \
    case 9: WT_BW_PICK(9, TT); break; \
    default: return nullptr;          \
  }
  if (dtype == 0) { WT_BW_PICK_K(float) }
  else if (dtype == 1) { WT_BW_PICK_K(__half) }
  else { WT_BW_PICK_K(__nv_bfloat16) }
#undef WT_BW_PICK_K
#undef WT_BW_PICK
  return f;
}

int bw_regs(int k, int mi, int dtype) {
  static std::mutex mu;
  static int cache[4][2][3];  // k = 3, 5, 7, 9; tiles per thread 1, 2; dtype; 0 = not yet read
  const int ki = (k - 3) / 2, mj = mi == 1 ? 0 : 1;
  if (ki < 0 || ki > 3 || dtype < 0 || dtype > 2) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[ki][mj][dtype] == 0) {
    WtBwPlan q;
    q.K = k;
    q.tbr = 4;
    q.mi = mi;
    const void* f = bw_pick(q, dtype);
    cudaFuncAttributes a;
    if (!f || cudaFuncGetAttributes(&a, f) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[ki][mj][dtype] = a.numRegs;
  }
  return cache[ki][mj][dtype];
}

// Resident parameter-gradient CTAs per SM for this plan (0 if the runtime
// cannot tell, e.g. without a device).
int bw_ctas_per_sm(const WtBwPlan& pl, int dtype) {
  const void* f = bw_pick(pl, dtype);
  if (!f) return 0;
  return occupancy(f, WT_BW_THREADS, pl.smem_bytes);
}

unsigned int take_bw_faults() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_bw_faults, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_bw_faults, &z, sizeof(z));
  return v;
}

}  // namespace wt
