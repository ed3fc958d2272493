// Fused WTConv2d backward (sm_103a): the input gradient and every parameter
// gradient from one read of x and dy.
//
// The two backward passes share their most expensive input: the Haar
// pyramid of dy.  The input gradient is the forward pass applied to dy with
// every kernel rotated by 180 degrees (A^T of the linear layer map), i.e.
// band convolutions of F_l dy and the collapsed synthesis plus the rotated
// base convolution.  The parameter gradients correlate the same F_l dy with
// F_l x.  A unit (channel, P planes) therefore loads x and dy once, builds
// both pyramids once, and then:
//   - correlates them into the per-thread accumulators (as the separate
//     parameter-gradient kernel: one record per (CTA, channel), finalized
//     in CTA order, so the result is deterministic);
//   - convolves the dy bands with the rotated, scale-folded level weights
//     into Z buffers;
//   - runs the final tiles (rotated base convolution on the dy plane +
//     bit-indexed synthesis) and stores dx.
// HBM traffic: x and dy read once, dx written once (3 element transfers
// instead of the 4 of the two separate passes).
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805), technical summary, "Key contributions"
// (all gradients reproduced by the fused implementation) and "Methodology"
// (analysis recomputed on chip, collapsed synthesis, folded scales).  The
// merging of the two backward passes into one kernel is this library's.
#pragma once

#include "wtconv_fwd_tiles.cuh"
#include "wtconv_launch.h"

namespace wt {

// Bounded waits that gave up; read by take_bwf_faults().
static __device__ unsigned int g_bwf_faults;

// TR: correlation tile rows (8: one tile per thread; the code also handles
// 4-row tiles, up to two per thread).  TP: final-tile height (level-1 rows)
// of the input-gradient tiles.  16-bit instances at k <= 5 are held to the
// registers of two CTAs per SM; the float32 ones are left to the compiler
// (0: no minimum), which fits those by itself (at k = 7, 9 the planner hands
// the layer to the two separate passes).
template <int K, typename T, int TR, int TP>
__global__ void __launch_bounds__(WT_BW_THREADS, sizeof(T) == 2 && K <= 5 ? 2 : 0)
    bwf_kernel(const __grid_constant__ WtBwPlan pl, const __grid_constant__ WtFwdPlan fp,
               const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmd,
               const T* __restrict__ x, const T* __restrict__ dy, const float* __restrict__ w_base,
               const float* __restrict__ w_sub, const float* __restrict__ s_base,
               const float* __restrict__ s_w, T* __restrict__ dx, float* __restrict__ part) {
  extern __shared__ __align__(16) float sm_raw[];
  float* const sm = align_smem128(sm_raw);  // box destinations need 128-byte alignment
  constexpr int KK = K * K;
  constexpr int NT = WT_BW_THREADS;
  constexpr int MI = TR == 8 ? 1 : WT_BW_MAX_ITEMS;
  constexpr int TC = 4;
  constexpr int ZT = WT_ZT;
  constexpr bool ASYNC = sizeof(T) == 4;
  constexpr int R = K / 2;
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L, P = pl.P, NB = pl.batches;
  const int u_begin = bw_unit_begin(pl, blockIdx.x);
  const int u_end = bw_unit_begin(pl, blockIdx.x + 1);
  const int c_first = fdiv(u_begin, pl.nb_div);
  const int XBF = pl.xbf, DBF = pl.dbf, WF = pl.wf;
  const int ipp = pl.items_per_plane;
  float* const work = sm + pl.work_off;
  float* const wsm = sm + fp.w_off;
  const int wb = fp.w_band;
  // Box path (float32, 16-byte rows): one thread issues the x and dy copies
  // of a unit into input set `s` (both planes with their margins: 4 columns
  // left, r rows above); both complete on mbar[s].
  const bool tma = ASYNC && pl.use_tma;
  const bool dbl = pl.nsets == 2;
  uint64_t* const mbar = reinterpret_cast<uint64_t*>(sm + pl.mb_off);
  __shared__ int s_ok;
  uint32_t parity = 0;  // thread 0: phase parity of mbar[0] (bit 0) and mbar[1] (bit 1)
  auto issue = [&](int u, int s) {
    const int cc = fdiv(u, pl.nb_div);
    const int n0 = (u - cc * NB) * P;
    float* const dst = sm + s * pl.islot;
    fence_proxy_async();  // earlier generic accesses of the set precede the copies
    mbar_arrive_expect_tx(&mbar[s], pl.tma_bytes + pl.dbg_extra_tx);
    tma_load_4d(dst, &tmx, -4, -R, cc, n0, &mbar[s]);
    tma_load_4d(dst + pl.xr, &tmd, -4, -R, cc, n0, &mbar[s]);
  };
  // Single input set: the x planes are last read by the correlations, the dy
  // planes by the final tiles, so the next unit's x box is requested as soon
  // as the correlations are done (issue_x, which also arms the barrier for
  // both boxes) and its dy box when the unit ends (issue_dy).
  auto issue_x = [&](int u) {
    const int cc = fdiv(u, pl.nb_div);
    const int n0 = (u - cc * NB) * P;
    fence_proxy_async();  // earlier generic accesses of the x planes precede the copy
    mbar_arrive_expect_tx(&mbar[0], pl.tma_bytes + pl.dbg_extra_tx);
    tma_load_4d(sm, &tmx, -4, -R, cc, n0, &mbar[0]);
  };
  auto issue_dy = [&](int u) {
    const int cc = fdiv(u, pl.nb_div);
    const int n0 = (u - cc * NB) * P;
    fence_proxy_async();  // earlier generic accesses of the dy planes precede the copy
    tma_load_4d(sm + pl.xr, &tmd, -4, -R, cc, n0, &mbar[0]);
  };
  auto prefetch = [&](int u) {  // the boxes issue(u, .) will copy, into L2
    const int cc = fdiv(u, pl.nb_div);
    const int n0 = (u - cc * NB) * P;
    tma_prefetch_4d(&tmx, -4, -R, cc, n0);
    tma_prefetch_4d(&tmd, -4, -R, cc, n0);
  };
  // 16-bit staged path (as in the parameter-gradient kernel): a unit's raw x
  // and dy planes land in the staging area (one bulk copy per plane on
  // mbar[0], or 8-byte cp.async chunks from every thread) and are widened
  // into the input set, after which the next unit's copies are issued.
  const bool bulk = !ASYNC && pl.use_bulk == 1;
  const bool cpa = !ASYNC && pl.use_bulk == 2;
  const bool staged = bulk || cpa;
  const int HWp = pl.H * pl.W;
  T* const stage_x = reinterpret_cast<T*>(sm + pl.stage_off);
  T* const stage_d = stage_x + P * HWp;
  auto issue_bulk = [&](int u) {
    const int cc = fdiv(u, pl.nb_div);
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
    const int cc = fdiv(u, pl.nb_div);
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

  // Zeroed once: interiors are rewritten per unit, margins stay zero.  The
  // work area is zeroed again after each channel's reduction, which reuses it.
  zero_smem(sm, pl.work_off + pl.red_floats, tid, NT);
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
  if (tma && tid == 0 && u_begin < u_end) issue(u_begin, 0);
  if (bulk && tid == 0 && u_begin < u_end) issue_bulk(u_begin);
  if (cpa && u_begin < u_end) issue_cpa(u_begin);

  int slot = 0;
  for (int u = u_begin; u < u_end;) {
    // The units of channel c held by this CTA: [u, u_stop).  The rotated,
    // folded weights of c are staged first (the previous unit and the
    // previous reduction ended with a barrier).
    const int c = fdiv(u, pl.nb_div);
    const int u_stop = min(u_end, (c + 1) * NB);
    stage_weights<K, true>(wsm, wb, L, C, c, w_base, w_sub, s_base, s_w, tid, NT);
    for (; u < u_stop; ++u, slot = dbl ? slot ^ 1 : 0) {
      const int n0 = (u - c * NB) * P;
      const int np = min(P, pl.N - n0);
      float* const in_x = sm + slot * pl.islot;  // this unit's x planes
      float* const in_d = in_x + pl.xr;          // ... and dy planes
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
      } else {
        load_planes<T>(in_x, XBF, pl.xs[0], x, n0, np, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
        load_planes<T>(in_d, DBF, pl.ds[0], dy, n0, np, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
      }
      __syncthreads();  // this unit's planes (and the weights) are visible
      if ((tma || bulk) && !s_ok) {  // the copy did not complete in time: record it and stop (uniform exit)
        const int mb = bulk ? 0 : slot;
        if (tid == 0) {
          atomicAdd(&g_bwf_faults, 1u);
          mbar_wait_bounded(&mbar[mb], ((parity >> mb) & 1u) ^ 1u, pl.wait_shift);  // let the copies in flight land
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

      // Both pyramids, once: levels 1+2 fused, then 3..L.
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

      // (a) Parameter-gradient correlations (one or two fixed tiles per thread).
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
            // One correlation instance serves every level: x's interior
            // starts pcol floats into a row (4 for the raw plane, 0 for the
            // bands, whose left margin is the previous row's right one), so
            // the window starts 4 - r floats after a 16-byte boundary.
            const WtBuf Xb = pl.xs[l], Db = pl.ds[l];
            const float* xb = l == 0 ? in_x + g * XBF : work + g * WF + b * Xb.band;
            const float* db = l == 0 ? in_d + g * DBF : work + g * WF + b * Db.band;
            const float sum = corr_tile<K, TR, TC, 4 - R>(xb + Xb.off + p0 * Xb.stride + q0 + Xb.pcol - 4, Xb.stride,
                                                          db + Db.off + (p0 + Db.prow) * Db.stride + q0 + Db.pcol,
                                                          Db.stride, acc[s]);
            if (l == 0) gs[s] += sum;
          }
        }
      }
      // (b) Input gradient, band convolutions: Z^l_b = conv(F_l dy, rotated
      // folded W_l,b), ZT x ZT tiles.  The dy bands' interiors start 4 floats
      // into each row, so a window starts 4 - r floats after a 16-byte boundary.
      for (int it = tid; it < np * fp.zipp; it += NT) {
        const int g = fdiv(it, fp.z_ipp);
        const int local = it - g * fp.zipp;
        int l = 1;
        while (l < L && local >= fp.zbegin[l + 1]) ++l;
        const int rel = local - fp.zbegin[l];
        const int b = fdiv(rel, fp.z_tiles[l]);
        const int t = rel - b * (fp.ztr[l] * fp.ztc[l]);
        const int tp = fdiv(t, fp.z_tc[l]);
        const int p0 = tp * ZT, q0 = (t - tp * fp.ztc[l]) * ZT;
        float* ps = work + g * WF;
        const WtBuf Yb = pl.ds[l];
        float z[ZT][ZT];
#pragma unroll
        for (int o = 0; o < ZT; ++o)
#pragma unroll
          for (int j = 0; j < ZT; ++j) z[o][j] = 0.f;
        conv_tile_off<K, ZT, ZT, 4 - R>(ps + Yb.off + b * Yb.band + (p0 - R + Yb.prow) * Yb.stride + q0 + Yb.pcol - 4,
                                        Yb.stride, wsm + (1 + 4 * (l - 1) + b) * wb, z);
        const WtBuf Zb = fp.zb[l];
        float* dst = ps + Zb.off + b * Zb.band + p0 * Zb.stride + q0;
        const int Hl = fp.Hs[l], Wl = fp.Ws[l];
        if (p0 + ZT <= Hl && q0 + ZT <= Wl) {
#pragma unroll
          for (int o = 0; o < ZT; ++o)
            *reinterpret_cast<float4*>(dst + o * Zb.stride) = make_float4(z[o][0], z[o][1], z[o][2], z[o][3]);
        } else {
#pragma unroll
          for (int o = 0; o < ZT; ++o)
#pragma unroll
            for (int j = 0; j < ZT; ++j)
              if (p0 + o < Hl && q0 + j < Wl) dst[o * Zb.stride + j] = z[o][j];
        }
      }
      __syncthreads();
      if (tma && !dbl && tid == 0 && u + 1 < u_end) issue_x(u + 1);  // single set: its x planes are free
      // (c) Input gradient, final tiles: rotated base convolution of the dy
      // plane + synthesis, stored to dx.
      final_tiles<K, T, TP, NT>(fp, work, in_d, wsm, 0.f, dx, n0, c, np, tid, 0, 0, 0, fp.H, fp.W);
      __syncthreads();  // every read of this unit is done
      if (tma && !dbl && tid == 0 && u + 1 < u_end) issue_dy(u + 1);  // single set: its dy planes are free
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
      zero_smem(work, pl.red_floats, tid, NT);  // restore the pyramids' and Z buffers' zero margins
      __syncthreads();
    }
  }
}

// The kernel for (k, dtype) with 8-row correlation tiles and half-height
// final tiles (for the planes that fit, at most 16 x 16 final tiles per
// plane, these never take more rounds of the 256 threads than full-height
// ones).
const void* bwf_kernel_tr8(int k, int dtype);
// Reads and clears the instantiating translation unit's fault counter.
unsigned int take_bwf_faults_tr8();

#define WT_BWF_INSTANTIATE(TRV)                                                                     \
  template <int K, typename T>                                                                      \
  static const void* bwf_fn_##TRV() {                                                               \
    return (const void*)bwf_kernel<K, T, TRV, WT_TP / 2>;                                           \
  }                                                                                                 \
  template <typename T>                                                                             \
  static const void* bwf_fn_k_##TRV(int k) {                                                        \
    switch (k) {                                                                                    \
      case 3: return bwf_fn_##TRV<3, T>();                                                          \
      case 5: return bwf_fn_##TRV<5, T>();                                                          \
      case 7: return bwf_fn_##TRV<7, T>();                                                          \
      case 9: return bwf_fn_##TRV<9, T>();                                                          \
      default: return nullptr;                                                                      \
    }                                                                                               \
  }                                                                                                 \
  const void* bwf_kernel_tr##TRV(int k, int dtype) {                                                \
    if (dtype == 0) return bwf_fn_k_##TRV<float>(k);                                                \
    if (dtype == 1) return bwf_fn_k_##TRV<__half>(k);                                               \
    return bwf_fn_k_##TRV<__nv_bfloat16>(k);                                                        \
  }                                                                                                 \
  unsigned int take_bwf_faults_tr##TRV() {                                                          \
    unsigned int v = 0, z = 0;                                                                      \
    if (cudaMemcpyFromSymbol(&v, g_bwf_faults, sizeof(v)) != cudaSuccess) return 0;                 \
    cudaMemcpyToSymbol(g_bwf_faults, &z, sizeof(z));                                                \
    return v;                                                                                       \
  }

}  // namespace wt
