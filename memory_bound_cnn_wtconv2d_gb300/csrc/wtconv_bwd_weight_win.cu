// WTConv2d parameter gradients for planes whose pyramids do not fit one CTA
// (sm_103a).
//
// The correlations behind every parameter gradient are sums over positions,
//   G_0[t]  = sum_{n,i,j} dy[i][j] * x[i+du-r][j+dv-r],   g = sum dy,
//   G_lb[t] = sum_{n,p,q} D^l_b[p][q] * Y^l_b[p+du-r][q+dv-r],
// (D^l = F_l dy, Y^l = F_l x), so they split over output tiles.  With tile
// origins at multiples of 2^L, a tile's dy coefficients D^l are built from
// the tile's own dy pixels, and the x coefficients Y^l they meet lie within r
// level-l positions of the tile, i.e. within 2^L * r input pixels.  A unit
// loads the dy tile and the x window (the tile plus that halo; zero outside
// the plane, which is the layer's zero extension), builds the pyramid of
// each, and correlates the tile's positions.  Positions of a ragged edge
// tile outside the plane have dy = 0 and add nothing.  Sums accumulate and
// reduce as in the whole-plane kernel: per-thread registers across a
// channel's units, one record per (CTA, channel), then the same
// deterministic finalize in CTA order.
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805), technical summary, "Key contributions"
// (every parameter gradient reproduced) and "Methodology" (scales folded into
// the weights, unfolded in the finalize).  The tiling is this library's.
#include <mutex>

#include "wtconv_device.cuh"
#include "wtconv_launch.h"

namespace wt {

// Bounded waits that gave up; read by take_bww_faults().
static __device__ unsigned int g_bww_faults;

// TR = 8: 8x4 correlation tiles, one per thread; TR = 4: 4x4, up to two.
template <int K, typename T, int TR>
__global__ void __launch_bounds__(WT_BW_THREADS)
    bw_win_kernel(const __grid_constant__ WtBwPlan pl, const __grid_constant__ CUtensorMap tmx,
                  const __grid_constant__ CUtensorMap tmd, const T* __restrict__ x, const T* __restrict__ dy,
                  float* __restrict__ part) {
  extern __shared__ __align__(16) float sm_raw[];
  float* const sm = align_smem128(sm_raw);  // box destinations need 128-byte alignment
  constexpr int KK = K * K;
  constexpr int NT = WT_BW_THREADS;
  constexpr int MI = TR == 8 ? 1 : WT_BW_MAX_ITEMS;
  constexpr int TC = 4;
  constexpr int R = K / 2;
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L, P = pl.P, NB = pl.batches;
  const int ntiles = pl.nty * pl.ntx;
  // Persistent CTA: an even share of the C * NB (channel, tile unit) list,
  // in order (channel, then plane group, then tile).
  const int u_begin = bw_unit_begin(pl, blockIdx.x);
  const int u_end = bw_unit_begin(pl, blockIdx.x + 1);
  const int c_first = fdiv(u_begin, pl.nb_div);
  const int XBF = pl.xbf, DBF = pl.dbf, WF = pl.wf;
  const int ipp = pl.items_per_plane;
  const int h = pl.halo, Hv = pl.Hs[0], Wv = pl.Ws[0], th = pl.th, tw = pl.tw;
  float* const work = sm + pl.work_off;
  const bool box32 = pl.win_load == 1;  // float32 boxes straight into an input set
  const bool box16 = pl.win_load == 2;  // 16-bit boxes into the staging area, widened per unit
  const bool boxed = box32 || box16;
  const bool dbl = box32 && pl.nsets == 2;
  uint64_t* const mbar = reinterpret_cast<uint64_t*>(sm + pl.mb_off);
  __shared__ int s_ok;
  uint32_t parity = 0;  // thread 0: phase parity of mbar[0] (bit 0) and mbar[1] (bit 1)
  const T* const stage_x = reinterpret_cast<const T*>(sm + pl.stage_off);
  const T* const stage_d = reinterpret_cast<const T*>(sm + pl.stage_off + pl.stage_dx);

  // Unit u -> channel, first plane, tile origin (the x window starts h
  // pixels above and left of it, negative at the top/left edge).
  auto decode = [&](int u, int& cc, int& n0, int& ty0, int& tx0) {
    cc = fdiv(u, pl.nb_div);
    const int rem = u - cc * NB;
    const int gi = rem / ntiles;
    const int t = rem - gi * ntiles;
    const int ty = t / pl.ntx;
    n0 = gi * P;
    ty0 = ty * th;
    tx0 = (t - ty * pl.ntx) * tw;
  };
  // One thread requests unit u: the x window box (float32: with the buffer's
  // margins, 4 columns left and r rows above) and the dy tile box, both
  // completing on mbar[s].  Every x coordinate is a multiple of 8 elements
  // (float32 x window: a multiple of 4 after the 4-column margin).
  auto issue = [&](int u, int s) {
    int cc, n0, ty0, tx0;
    decode(u, cc, n0, ty0, tx0);
    fence_proxy_async();  // earlier generic accesses of the destinations precede the copies
    mbar_arrive_expect_tx(&mbar[s], pl.tma_bytes + pl.dbg_extra_tx);
    if (box32) {
      float* const dst = sm + s * pl.islot;
      tma_load_4d(dst, &tmx, tx0 - h - 4, ty0 - h - R, cc, n0, &mbar[s]);
      tma_load_4d(dst + pl.xr, &tmd, tx0, ty0, cc, n0, &mbar[s]);
    } else {
      tma_load_4d(sm + pl.stage_off, &tmx, tx0 - h, ty0 - h, cc, n0, &mbar[s]);
      tma_load_4d(sm + pl.stage_off + pl.stage_dx, &tmd, tx0, ty0, cc, n0, &mbar[s]);
    }
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
  if (boxed && tid == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (boxed && tid == 0 && u_begin < u_end) issue(u_begin, 0);

  int slot = 0;
  for (int u = u_begin; u < u_end;) {
    // The units of channel c held by this CTA: [u, u_stop).
    const int c = fdiv(u, pl.nb_div);
    const int u_stop = min(u_end, (c + 1) * NB);
    for (; u < u_stop; ++u, slot = dbl ? slot ^ 1 : 0) {
      int cc, n0, ty0, tx0;
      decode(u, cc, n0, ty0, tx0);
      const int np = min(P, pl.N - n0);
      float* const in_x = sm + slot * pl.islot;  // this unit's x windows
      float* const in_d = in_x + pl.xr;          // ... and dy tiles
      if (boxed) {
        if (tid == 0) {
          const bool ok = mbar_wait_bounded(&mbar[slot], (parity >> slot) & 1u, pl.wait_shift);
          parity ^= 1u << slot;
          if (ok && dbl && u + 1 < u_end) issue(u + 1, slot ^ 1);  // the other set was last read by unit u-1
          s_ok = ok;
        }
      } else {
        load_window<T>(in_x, XBF, pl.xs[0], x, n0, np, c, C, pl.H, pl.W, ty0 - h, tx0 - h, Hv, Wv, pl.vec_ok != 0,
                       pl.ld_pp, pl.ld_w, tid, NT);
        load_window<T>(in_d, DBF, pl.ds[0], dy, n0, np, c, C, pl.H, pl.W, ty0, tx0, th, tw, pl.vec_ok != 0,
                       pl.dld_pp, pl.dld_w, tid, NT);
      }
      __syncthreads();  // this unit's windows and tiles are visible
      if (boxed && !s_ok) {  // the copy did not complete in time: record it and stop (uniform exit)
        if (tid == 0) {
          atomicAdd(&g_bww_faults, 1u);
          mbar_wait_bounded(&mbar[slot], ((parity >> slot) & 1u) ^ 1u, pl.wait_shift);  // let the copies in flight land
        }
        __syncthreads();
        return;  // records are not written: the caller sees the fault count
      }
      if (box16) {  // widen the raw windows and tiles, then request the next unit's
        widen_planes<T>(in_x, XBF, pl.xs[0], stage_x, np, Hv, Wv, 4, pl.wd_pp, pl.wd_w, tid, NT);
        widen_planes<T>(in_d, DBF, pl.ds[0], stage_d, np, th, tw, 4, pl.dwd_pp, pl.dwd_w, tid, NT);
        __syncthreads();
        if (tid == 0 && u + 1 < u_end) issue(u + 1, 0);
      }

      // Pyramids: the x window's and the dy tile's (levels 1+2 fused, then 3..L).
      if (L == 1) {
        haar_level(in_x, XBF, work, WF, np, pl.xs[0], pl.xs[1], pl.Hs[1], pl.Ws[1], pl.an_pp[1], pl.an_w[1], tid, NT);
        haar_level(in_d, DBF, work, WF, np, pl.ds[0], pl.ds[1], pl.dHs[1], pl.dWs[1], pl.dn_pp[1], pl.dn_w[1], tid,
                   NT);
      } else {
        haar_levels12(in_x, XBF, work, WF, np, pl.xs[0], pl.xs[1], pl.xs[2], pl.Hs[1], pl.Ws[1], pl.Hs[2], pl.Ws[2],
                      pl.an_pp[2], pl.an_w[2], tid, NT);
        haar_levels12(in_d, DBF, work, WF, np, pl.ds[0], pl.ds[1], pl.ds[2], pl.dHs[1], pl.dWs[1], pl.dHs[2],
                      pl.dWs[2], pl.dn_pp[2], pl.dn_w[2], tid, NT);
      }
      __syncthreads();
      for (int l = 3; l <= L; ++l) {
        haar_level(work, WF, work, WF, np, pl.xs[l - 1], pl.xs[l], pl.Hs[l], pl.Ws[l], pl.an_pp[l], pl.an_w[l], tid,
                   NT);
        haar_level(work, WF, work, WF, np, pl.ds[l - 1], pl.ds[l], pl.dHs[l], pl.dWs[l], pl.dn_pp[l], pl.dn_w[l], tid,
                   NT);
        __syncthreads();
      }

      // Correlations over the tile: TR x 4 tiles at tile-relative (p0, q0),
      // against the x window from position (zo + p0 - r, zo + q0 - r); the
      // level buffers' column margin puts each window row on a 16-byte
      // boundary.  Rows of a level's last tile row past the tile read dy = 0.
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
            // One instance for every level: the tile's origin sits zo floats
            // into the level's window interior (h for the raw window), which
            // starts pcol floats into a row with zo + pcol a multiple of 4, so
            // the correlation window starts 4 - r floats after a 16-byte
            // boundary.  The dy tile and its bands have no margins.
            const WtBuf Xb = pl.xs[l], Db = pl.ds[l];
            const int zo = pl.zo[l];
            const float* xb = l == 0 ? in_x + g * XBF : work + g * WF + b * Xb.band;
            const float* db = l == 0 ? in_d + g * DBF : work + g * WF + b * Db.band;
            const float sum = corr_tile<K, TR, TC, 4 - R>(
                xb + Xb.off + (zo + p0 - R + Xb.prow) * Xb.stride + zo + q0 + Xb.pcol - 4, Xb.stride,
                db + Db.off + p0 * Db.stride + q0, Db.stride, acc[s]);
            if (l == 0) gs[s] += sum;
          }
        }
      }
      __syncthreads();  // every read of this unit is done
      if (box32 && !dbl && tid == 0 && u + 1 < u_end) issue(u + 1, 0);  // single set: refill it now
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

template <int K, typename T>
static const void* bw_win_fn(int tbr) {
  return tbr == 8 ? (const void*)bw_win_kernel<K, T, 8> : (const void*)bw_win_kernel<K, T, 4>;
}

template <typename T>
static const void* bw_win_fn_k(int k, int tbr) {
  switch (k) {
    case 3: return bw_win_fn<3, T>(tbr);
    case 5: return bw_win_fn<5, T>(tbr);
    case 7: return bw_win_fn<7, T>(tbr);
    case 9: return bw_win_fn<9, T>(tbr);
    default: return nullptr;
  }
}

static const void* bw_win_pick(const WtBwPlan& pl, int dtype) {
  if (dtype == 0) return bw_win_fn_k<float>(pl.K, pl.tbr);
  if (dtype == 1) return bw_win_fn_k<__half>(pl.K, pl.tbr);
  return bw_win_fn_k<__nv_bfloat16>(pl.K, pl.tbr);
}

cudaError_t launch_bwd_weight_win(const WtBwPlan& pl, const CUtensorMap& tmx, const CUtensorMap& tmd, int dtype,
                                  const void* x, const void* dy, const float* w_base, const float* b_base,
                                  const float* w_sub, const float* s_base, const float* s_w, float* dw_base,
                                  float* db_base, float* dw_sub, float* ds_base, float* ds_w, float* part,
                                  cudaStream_t stream) {
  const void* f = bw_win_pick(pl, dtype);
  if (!f) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(f, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  WtBwPlan plc = pl;
  CUtensorMap mx = tmx, md = tmd;
  void* args[] = {(void*)&plc, (void*)&mx, (void*)&md, (void*)&x, (void*)&dy, (void*)&part};
  e = cudaLaunchKernel(f, dim3((unsigned)pl.grid), dim3(WT_BW_THREADS), args, (size_t)pl.smem_bytes, stream);
  if (e != cudaSuccess) return e;
  return launch_bw_finalize(pl, part, w_base, b_base, w_sub, s_base, s_w, dw_base, db_base, dw_sub, ds_base, ds_w,
                            stream);
}

int bw_win_regs(int k, int tbr, int dtype) {
  static std::mutex mu;
  static int cache[4][2][3];  // k = 3, 5, 7, 9; tbr = 8, 4; dtype; 0 = not yet read
  const int ki = (k - 3) / 2, ti = tbr == 8 ? 0 : 1;
  if (ki < 0 || ki > 3 || dtype < 0 || dtype > 2) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[ki][ti][dtype] == 0) {
    WtBwPlan q;
    q.K = k;
    q.tbr = tbr;
    const void* f = bw_win_pick(q, dtype);
    cudaFuncAttributes a;
    if (!f || cudaFuncGetAttributes(&a, f) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[ki][ti][dtype] = a.numRegs;
  }
  return cache[ki][ti][dtype];
}

int bw_win_ctas_per_sm(const WtBwPlan& pl, int dtype) {
  const void* f = bw_win_pick(pl, dtype);
  if (!f) return 0;
  return occupancy(f, WT_BW_THREADS, pl.smem_bytes);
}

unsigned int take_bww_faults() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_bww_faults, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_bww_faults, &z, sizeof(z));
  return v;
}

}  // namespace wt
