// Windowed forward / input-gradient pass for planes whose Haar pyramid does
// not fit one CTA's shared memory (sm_103a).
//
// The output plane is cut into th x tw tiles whose origins are multiples of
// 2^L.  Output (i, j) reads, from every level l, the convolved coefficients at
// (i >> l, j >> l); the k x k band convolution reaches r coefficients further,
// and a level-l coefficient is built from one 2^l x 2^l input block.  A tile
// therefore depends on the input within 2^L * r pixels of it (r for the base
// convolution).  A unit loads the tile's window with a halo h >= 2^L * r that
// is a multiple of 2^L, so the window's Haar blocks are the plane's own
// blocks, and pixels outside the plane read as zero, which is the layer's own
// zero extension of odd sizes and its "same" padding.  The CTA builds the
// pyramid of the whole window, convolves the bands at the tile's
// coefficients only (all of whose k x k neighbourhoods lie inside the
// window), and runs the same final tiles as the whole-plane kernel.  Every
// output is therefore the same sum of the same coefficients as there.
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805), technical summary, "Methodology" (the
// analysis recomputed on chip, the collapsed synthesis, the folded scales).
// The pages describe the fused kernels, not how planes larger than on-chip
// memory are split; the halo tiling is this library's.
#include "wtconv_fwd_tiles.cuh"
#include "wtconv_launch.h"

namespace wt {

// Bounded waits that gave up; read by take_win_faults().
static __device__ unsigned int g_win_faults;

// Persistent: CTA b owns the units [b*U/G, (b+1)*U/G) of the unit list,
// ordered by channel, then plane group, then tile (row-major), so
// consecutive units usually share a channel and its folded weights.
template <int K, typename T, bool ROT>
__global__ void __launch_bounds__(WT_FWD_THREADS, 3)
    fwd_win_kernel(const __grid_constant__ WtFwdPlan pl, const __grid_constant__ CUtensorMap tmx,
                   const T* __restrict__ x, const float* __restrict__ w_base, const float* __restrict__ b_base,
                   const float* __restrict__ w_sub, const float* __restrict__ s_base,
                   const float* __restrict__ s_w, T* __restrict__ y) {
  extern __shared__ __align__(16) float sm_raw[];
  float* const sm = align_smem128(sm_raw);  // box destinations need 128-byte alignment
  constexpr int R = K / 2;
  constexpr int NT = WT_FWD_THREADS;
  constexpr int ZT = WT_ZT;
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L, P = pl.P;
  const int XF = pl.xf, WF = pl.wf;
  const int ntiles = pl.nty * pl.ntx;
  const int per_c = pl.groups * ntiles;
  const long long units = (long long)C * per_c;
  const int u_begin = (int)(units * blockIdx.x / gridDim.x);
  const int u_end = (int)(units * (blockIdx.x + 1) / gridDim.x);
  float* const wsm = sm + pl.w_off;
  float* const work = sm + pl.work_off;
  const int wb = pl.w_band;
  const int Hv = pl.Hs[0], Wv = pl.Ws[0];
  const bool box32 = pl.win_load == 1;  // float32 window boxes straight into an input set
  const bool box16 = pl.win_load == 2;  // 16-bit window boxes into the staging area
  const bool boxed = box32 || box16;
  const bool dbl = box32 && pl.nsets == 2;
  uint64_t* const mbar = reinterpret_cast<uint64_t*>(sm + pl.mb_off);
  __shared__ int s_ok;
  uint32_t parity = 0;  // thread 0: current phase parity of mbar[0] (bit 0) and mbar[1] (bit 1)

  // Unit uu -> channel, first plane, window origin (negative at the top/left edge).
  auto decode = [&](int uu, int& cc, int& nn, int& oy, int& ox) {
    cc = uu / per_c;
    const int rem = uu - cc * per_c;
    const int gi = rem / ntiles;
    const int t = rem - gi * ntiles;
    const int ty = t / pl.ntx;
    nn = gi * P;
    oy = ty * pl.th - pl.halo;
    ox = (t - ty * pl.ntx) * pl.tw - pl.halo;
  };
  // One thread requests unit uu's windows: float32 boxes land in input set s
  // with the buffer's margins (4 columns left, r rows above; ox - 4 is a
  // multiple of 4), 16-bit boxes land raw in the staging area (ox a multiple
  // of 8).  Both complete on mbar[s]; pixels outside the tensor read as zero.
  auto issue = [&](int uu, int s) {
    int cc, nn, oy, ox;
    decode(uu, cc, nn, oy, ox);
    fence_proxy_async();  // earlier generic accesses of the destination precede the copy
    mbar_arrive_expect_tx(&mbar[s], pl.tma_bytes + pl.dbg_extra_tx);
    if (box32) tma_load_4d(sm + s * pl.xslot, &tmx, ox - 4, oy - R, cc, nn, &mbar[s]);
    else tma_load_4d(sm + pl.stage_off, &tmx, ox, oy, cc, nn, &mbar[s]);
  };

  zero_smem(sm, pl.w_off, tid, NT);  // margins of every buffer stay zero (later writes touch interiors)
  if (boxed && tid == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();  // the zero fill and barrier init land before any copy
  if (boxed && tid == 0 && u_begin < u_end) issue(u_begin, 0);
  int c_prev = -1;
  int slot = 0;
  for (int u = u_begin; u < u_end; ++u, slot = dbl ? slot ^ 1 : 0) {
    int c, n0, oy, ox;
    decode(u, c, n0, oy, ox);
    const int np = min(P, pl.N - n0);
    float* const xs = sm + slot * pl.xslot;
    if (c != c_prev) {
      stage_weights<K, ROT>(wsm, wb, L, C, c, w_base, w_sub, s_base, s_w, tid, NT);
      c_prev = c;
    }
    if (boxed) {
      if (tid == 0) {
        if (box32 && !dbl && u != u_begin) issue(u, 0);  // single set: the previous unit is done with it
        const bool ok = mbar_wait_bounded(&mbar[slot], (parity >> slot) & 1u, pl.wait_shift);
        parity ^= 1u << slot;
        if (ok && dbl && u + 1 < u_end) issue(u + 1, slot ^ 1);  // the other set was last read by unit u-1
        s_ok = ok;
      }
    } else {
      load_window<T>(xs, XF, pl.lev[0], x, n0, np, c, C, pl.H, pl.W, oy, ox, Hv, Wv, pl.vec_ok != 0, pl.ld_pp,
                     pl.ld_w, tid, NT);
    }
    const float bias = (!ROT && b_base != nullptr) ? s_base[c] * b_base[c] : 0.f;
    __syncthreads();  // windows of unit u and the weights are visible
    if (boxed && !s_ok) {  // the copy did not complete in time: record it and stop (uniform exit)
      if (tid == 0) {
        atomicAdd(&g_win_faults, 1u);
        mbar_wait_bounded(&mbar[slot], ((parity >> slot) & 1u) ^ 1u, pl.wait_shift);  // let the copy in flight land
      }
      __syncthreads();
      break;
    }
    if (box16) {  // widen the raw windows, then request the next unit's
      widen_planes<T>(xs, XF, pl.lev[0], reinterpret_cast<const T*>(sm + pl.stage_off), np, Hv, Wv, 4,
                      pl.wd_pp, pl.wd_w, tid, NT);
      __syncthreads();
      if (tid == 0 && u + 1 < u_end) issue(u + 1, 0);
    }

    // (1) Haar pyramid of the whole window.
    if (L == 1) {
      haar_level(xs, XF, work, WF, np, pl.lev[0], pl.lev[1], pl.Hs[1], pl.Ws[1], pl.an_pp[1], pl.an_w[1], tid, NT);
    } else {
      haar_levels12(xs, XF, work, WF, np, pl.lev[0], pl.lev[1], pl.lev[2], pl.Hs[1], pl.Ws[1], pl.Hs[2],
                    pl.Ws[2], pl.an_pp[2], pl.an_w[2], tid, NT);
    }
    __syncthreads();
    for (int l = 3; l <= L; ++l) {
      haar_level(work, WF, work, WF, np, pl.lev[l - 1], pl.lev[l], pl.Hs[l], pl.Ws[l], pl.an_pp[l], pl.an_w[l],
                 tid, NT);
      __syncthreads();
    }

    // Band convolutions at the tile's coefficients: ZT x ZT tiles at
    // tile-relative (p0, q0), read from window position (zo + p0, zo + q0);
    // the level buffers' column margin makes every read row start 16-byte
    // aligned.
    for (int it = tid; it < np * pl.zipp; it += NT) {
      const int g = fdiv(it, pl.z_ipp);
      const int local = it - g * pl.zipp;
      int l = 1;
      while (l < L && local >= pl.zbegin[l + 1]) ++l;
      const int rel = local - pl.zbegin[l];
      const int b = fdiv(rel, pl.z_tiles[l]);
      const int t = rel - b * (pl.ztr[l] * pl.ztc[l]);
      const int tp = fdiv(t, pl.z_tc[l]);
      const int p0 = tp * ZT, q0 = (t - tp * pl.ztc[l]) * ZT;
      const int zo = pl.zo[l];
      float* ps = work + g * WF;
      const WtBuf Yb = pl.lev[l];
      float z[ZT][ZT];
#pragma unroll
      for (int o = 0; o < ZT; ++o)
#pragma unroll
        for (int j = 0; j < ZT; ++j) z[o][j] = 0.f;
      conv_tile<K, ZT, ZT>(ps + Yb.off + b * Yb.band + (zo + p0 - R + Yb.prow) * Yb.stride + zo + q0 - R + Yb.pcol,
                           Yb.stride, wsm + (1 + 4 * (l - 1) + b) * wb, z);
      const WtBuf Zb = pl.zb[l];
      float* dst = ps + Zb.off + b * Zb.band + p0 * Zb.stride + q0;
      const int Tl = pl.th >> l, Ul = pl.tw >> l;
      if (p0 + ZT <= Tl && q0 + ZT <= Ul) {
#pragma unroll
        for (int o = 0; o < ZT; ++o)
          *reinterpret_cast<float4*>(dst + o * Zb.stride) = make_float4(z[o][0], z[o][1], z[o][2], z[o][3]);
      } else {
#pragma unroll
        for (int o = 0; o < ZT; ++o)
#pragma unroll
          for (int j = 0; j < ZT; ++j)
            if (p0 + o < Tl && q0 + j < Ul) dst[o * Zb.stride + j] = z[o][j];
      }
    }
    __syncthreads();

    // (2) final tiles of the output tile (window offset h, plane origin oy + h, ox + h).
    const int h = pl.halo;
    if (pl.ftp == WT_TP)
      final_tiles<K, T, WT_TP>(pl, work, xs, wsm, bias, y, n0, c, np, tid, h, oy + h, ox + h, pl.H, pl.W);
    else
      final_tiles<K, T, WT_TP / 2>(pl, work, xs, wsm, bias, y, n0, c, np, tid, h, oy + h, ox + h, pl.H, pl.W);
    __syncthreads();  // all reads of unit u are done
  }  // unit loop
}

template <int K, typename T, bool ROT>
static cudaError_t launch_win_t(const WtFwdPlan& pl, const CUtensorMap& tmx, const void* x, const float* w_base,
                                const float* b_base, const float* w_sub, const float* s_base,
                                const float* s_w, void* y, cudaStream_t stream) {
  auto kern = fwd_win_kernel<K, T, ROT>;
  cudaError_t e = ensure_smem((const void*)kern, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  const int per_sm = occupancy((const void*)kern, WT_FWD_THREADS, pl.smem_bytes);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const long long units = (long long)pl.C * pl.groups * pl.nty * pl.ntx;
  long long slots = (long long)(per_sm < 1 ? 1 : per_sm) * sms;
  const unsigned grid = (unsigned)(units < slots ? units : slots);
  kern<<<grid, WT_FWD_THREADS, pl.smem_bytes, stream>>>(pl, tmx, static_cast<const T*>(x), w_base, b_base,
                                                        w_sub, s_base, s_w, static_cast<T*>(y));
  return cudaGetLastError();
}

template <typename T, bool ROT>
static cudaError_t launch_win_k(const WtFwdPlan& pl, const CUtensorMap& tmx, const void* x,
                                const float* w_base, const float* b_base, const float* w_sub,
                                const float* s_base, const float* s_w, void* y, cudaStream_t stream) {
  switch (pl.K) {
    case 3: return launch_win_t<3, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 5: return launch_win_t<5, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 7: return launch_win_t<7, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 9: return launch_win_t<9, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd_win(const WtFwdPlan& pl, const CUtensorMap& tmx, int dtype, bool rotate, const void* x,
                           const float* w_base, const float* b_base, const float* w_sub, const float* s_base,
                           const float* s_w, void* y, cudaStream_t stream) {
  if (dtype == 0)
    return rotate ? launch_win_k<float, true>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_win_k<float, false>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  if (dtype == 1)
    return rotate ? launch_win_k<__half, true>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_win_k<__half, false>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  return rotate ? launch_win_k<__nv_bfloat16, true>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                : launch_win_k<__nv_bfloat16, false>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
}

unsigned int take_win_faults() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_win_faults, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_win_faults, &z, sizeof(z));
  return v;
}

}  // namespace wt
