// Fused WTConv2d forward pass and input-gradient pass (sm_103a).
//
// A persistent grid walks units of P planes of one channel.  The planes
// cross HBM once: they are read into shared memory, the Haar pyramid is
// rebuilt there, every band of every level is convolved with scale-folded
// weights, and the final tiles add the base convolution and the synthesis of
// all levels in registers and write the output directly.
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805), technical summary, "Methodology":
//  (1) the Haar analysis butterflies are recomputed on chip instead of
//      writing the coefficient tensors Y^(l) to HBM;
//  (2) the L-step synthesis loop is replaced by the closed-form bit-indexed
//      sum ("Proposition 2"): output (i, j) receives, from every level l,
//      sum_b sign_b(bit_{l-1}(i), bit_{l-1}(j)) * Z^l_b[i >> l][j >> l];
//  (3) the per-channel scales are folded into the convolution weights (and
//      the base scale into the bias).
// The 2^-l normalisations of analysis and synthesis (4^-l in total) are also
// folded into the level-l weights, so every butterfly is a pure add.
//
// Phases per unit (one CTA barrier after each):
//   load (TMA / bulk / cp.async, the next unit prefetched where the layout
//   allows) -> Haar levels 1+2 (fused) -> Haar levels 3..L -> band
//   convolutions of all levels (Z buffers) -> final tiles (base conv + (2),
//   stored to HBM).
//
// The input-gradient pass is the same kernel with every kernel rotated by
// 180 degrees and no bias: the layer map is A = s_b*Conv_b + sum_l F_l^T K_l F_l
// with orthonormal F_l, so A^T = s_b*Conv_b^T + sum_l F_l^T K_l^T F_l and the
// transpose of a same-padded odd-k correlation is the correlation with the
// rotated kernel.
#include "wtconv_fwd_tiles.cuh"
#include "wtconv_launch.h"

#include <mutex>

namespace wt {

// Bounded waits that gave up (see mbar_wait_bounded); read by take_fwd_faults().
static __device__ unsigned int g_fwd_faults;

// Persistent: CTA b owns the units [b*U/G, (b+1)*U/G) of the channel-major
// unit list (unit = P planes of one channel), so consecutive units usually
// share a channel and its folded weights.  Shared memory holds two sets of
// input-plane buffers (the next unit's planes are prefetched with cp.async
// while the current unit is computed, for float32), one work area per plane
// (pyramid + convolved bands) and the weights.  It is zeroed once; later
// writes touch interiors only, so every margin stays zero.  Registers: at
// most 128 per thread for k <= 5 (no spills), so four CTAs fit an SM when a
// unit's shared memory allows it (small planes); 170 for k = 7, 9 (three).
template <int K, typename T, bool ROT>
__global__ void __launch_bounds__(WT_FWD_THREADS, K <= 5 ? 4 : 3)
    fwd_kernel(const __grid_constant__ WtFwdPlan pl, const __grid_constant__ CUtensorMap tmx,
               const T* __restrict__ x,
               const float* __restrict__ w_base, const float* __restrict__ b_base,
               const float* __restrict__ w_sub, const float* __restrict__ s_base,
               const float* __restrict__ s_w, T* __restrict__ y) {
  extern __shared__ __align__(16) float sm_raw[];
  float* const sm = align_smem128(sm_raw);  // TMA box destinations need 128-byte alignment
  constexpr int R = K / 2;
  constexpr int NT = WT_FWD_THREADS;
  constexpr int ZT = WT_ZT;
  constexpr bool ASYNC = sizeof(T) == 4;
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L;
  const int XF = pl.xf, WF = pl.wf;
  const long long units = (long long)C * pl.groups;
  const int u_begin = (int)(units * blockIdx.x / gridDim.x);
  const int u_end = (int)(units * (blockIdx.x + 1) / gridDim.x);
  float* const wsm = sm + pl.w_off;
  float* const work = sm + pl.work_off;
  const int wb = pl.w_band;

  // TMA path (float32, 16-byte rows): one thread issues one box copy per
  // unit into the input buffer set `slot`; the copy engine writes the whole
  // padded box (margins zero-filled) and completes on mbar[slot].
  const bool tma = ASYNC && pl.use_tma;
  uint64_t* const mbar = reinterpret_cast<uint64_t*>(sm + pl.mb_off);
  __shared__ int s_ok;
  uint32_t parity = 0;  // thread 0: current phase parity of mbar[0] (bit 0) and mbar[1] (bit 1)
  auto issue = [&](int uu, int s) {
    const int cc = uu / pl.groups;
    const int nn = (uu - cc * pl.groups) * pl.P;
    fence_proxy_async();  // earlier generic accesses of the buffer set precede the copy
    mbar_arrive_expect_tx(&mbar[s], pl.tma_bytes + pl.dbg_extra_tx);
    tma_load_4d(sm + s * pl.xslot, &tmx, -4, -R, cc, nn, &mbar[s]);
  };
  auto prefetch = [&](int uu) {  // the box issue(uu, .) will copy, into L2
    const int cc = uu / pl.groups;
    const int nn = (uu - cc * pl.groups) * pl.P;
    tma_prefetch_4d(&tmx, -4, -R, cc, nn);
  };
  // 16-bit staged path: the raw planes of a unit land in the staging area
  // after the first input set (one bulk copy per plane on mbar[0], or 8-byte
  // cp.async chunks from every thread); they are widened into the first set at
  // the start of the unit, after which the next unit's copies are issued.
  const bool bulk = !ASYNC && pl.use_bulk == 1;
  const bool cpa = !ASYNC && pl.use_bulk == 2;  // same staging, filled by every thread's 8-byte cp.async
  const bool staged = bulk || cpa;
  T* const stage = reinterpret_cast<T*>(sm + pl.stage_off);
  const int HWp = pl.H * pl.W;
  auto issue_bulk = [&](int uu) {
    const int cc = uu / pl.groups;
    const int nn = (uu - cc * pl.groups) * pl.P;
    const int npp = min(pl.P, pl.N - nn);
    fence_proxy_async();  // the widening reads of the staging area precede the copies
    mbar_arrive_expect_tx(&mbar[0], (uint32_t)npp * pl.bulk_bytes + pl.dbg_extra_tx);
    for (int g = 0; g < npp; ++g)
      bulk_load(stage + g * HWp, x + ((size_t)(nn + g) * C + cc) * HWp, pl.bulk_bytes, &mbar[0]);
  };
  auto issue_cpa = [&](int uu) {
    const int cc = uu / pl.groups;
    const int nn = (uu - cc * pl.groups) * pl.P;
    const int chunks = HWp >> 2;  // 8-byte chunks (4 elements) per plane
    const int total = min(pl.P, pl.N - nn) * chunks;
    for (int i = tid; i < total; i += NT) {
      const int g = fdiv(i, pl.cp_pp);
      const int o = (i - g * chunks) << 2;
      cp_async8(reinterpret_cast<float*>(stage + g * HWp + o),
                reinterpret_cast<const float*>(x + ((size_t)(nn + g) * C + cc) * HWp + o));
    }
    cp_async_commit();
  };

  // Zero margins once (the box copies write whole padded planes themselves).
  if (tma) zero_smem(sm + pl.work_off, pl.w_off - pl.work_off, tid, NT);
  else zero_smem(sm, pl.w_off, tid, NT);
  if ((tma || bulk) && tid == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();  // the zero fill and barrier init land before any plane copy
  if (tma && tid == 0 && u_begin < u_end) issue(u_begin, 0);
  if (bulk && tid == 0 && u_begin < u_end) issue_bulk(u_begin);
  if (cpa && u_begin < u_end) issue_cpa(u_begin);
  int c_prev = -1;
  float bias = 0.f;  // folded bias of channel c_prev
  int slot = 0;
  const bool dbl = pl.nsets == 2;
  for (int u = u_begin; u < u_end; ++u, slot = (dbl && !staged) ? slot ^ 1 : 0) {
    const int c = u / pl.groups;
    const int n0 = (u - c * pl.groups) * pl.P;
    const int np = min(pl.P, pl.N - n0);
    float* const xs = sm + slot * pl.xslot;
    if (c != c_prev) {
      stage_weights<K, ROT>(wsm, wb, L, C, c, w_base, w_sub, s_base, s_w, tid, NT);
      bias = (!ROT && b_base != nullptr) ? s_base[c] * b_base[c] : 0.f;
      c_prev = c;
    }
    if (tma) {
      if (tid == 0) {
        if (!dbl && u != u_begin) issue(u, 0);  // single set: the previous unit is done with it
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
    } else if (!ASYNC) {
      load_planes<T>(xs, XF, pl.lev[0], x, n0, np, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
    } else {
      if (u == u_begin || !dbl) {  // first unit, or single set: load now
        load_planes_async(xs, XF, pl.lev[0], reinterpret_cast<const float*>(x), n0, np, c, C, pl.H, pl.W,
                          pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
        cp_async_commit();
        cp_async_wait_all();
      }
      if (dbl && u + 1 < u_end) {  // prefetch the next unit into the other buffer set
        const int c1 = (u + 1) / pl.groups;
        const int n1 = (u + 1 - c1 * pl.groups) * pl.P;
        load_planes_async(sm + (slot ^ 1) * pl.xslot, XF, pl.lev[0], reinterpret_cast<const float*>(x), n1,
                          min(pl.P, pl.N - n1), c1, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
        cp_async_commit();
      }
    }
    __syncthreads();  // planes of unit u and the weights are visible
    if ((tma || bulk) && !s_ok) {  // the copy did not complete in time: record it and stop (uniform exit)
      const int mb = bulk ? 0 : slot;
      if (tid == 0) {
        atomicAdd(&g_fwd_faults, 1u);
        mbar_wait_bounded(&mbar[mb], ((parity >> mb) & 1u) ^ 1u, pl.wait_shift);  // let the copy in flight land
      }
      __syncthreads();
      break;
    }
    // 16-bit raw planes: widened by the fused level-1/2 pass itself where rows
    // have even length (4-element groups or pairs; 1-3 % faster at 14 x 14,
    // 28 x 28 and 56 x 56), else first, by a pass of their own.  The next
    // unit's copy follows once they are consumed.
    const bool widen12 = staged && L >= 2 && (pl.W & 1) == 0;
    if (staged && !widen12) {
      widen_planes<T>(xs, XF, pl.lev[0], stage, np, pl.H, pl.W, pl.wd_vec, pl.wd_pp, pl.wd_w, tid, NT);
      __syncthreads();
      if (bulk && tid == 0 && u + 1 < u_end) issue_bulk(u + 1);
      if (cpa && u + 1 < u_end) issue_cpa(u + 1);
    }

    // (1) Haar pyramid on chip.
    if (L == 1) {
      haar_level(xs, XF, work, WF, np, pl.lev[0], pl.lev[1], pl.Hs[1], pl.Ws[1], pl.an_pp[1], pl.an_w[1], tid, NT);
    } else if (widen12) {
      if constexpr (!ASYNC)  // (16-bit instances only)
        widen_levels12<T>(stage, pl.H, pl.W, xs, XF, pl.lev[0], work, WF, np, pl.lev[1], pl.lev[2], pl.Hs[1],
                          pl.Ws[1], pl.Hs[2], pl.Ws[2], pl.an_pp[2], pl.an_w[2], tid, NT);
    } else {
      haar_levels12(xs, XF, work, WF, np, pl.lev[0], pl.lev[1], pl.lev[2], pl.Hs[1], pl.Ws[1], pl.Hs[2],
                    pl.Ws[2], pl.an_pp[2], pl.an_w[2], tid, NT);
    }
    __syncthreads();
    if (widen12) {  // the raw planes are consumed: start the next unit's copy
      if (bulk && tid == 0 && u + 1 < u_end) issue_bulk(u + 1);
      if (cpa && u + 1 < u_end) issue_cpa(u + 1);
    }
    for (int l = 3; l <= L; ++l) {
      haar_level(work, WF, work, WF, np, pl.lev[l - 1], pl.lev[l], pl.Hs[l], pl.Ws[l], pl.an_pp[l], pl.an_w[l],
                 tid, NT);
      __syncthreads();
    }

    // Band convolutions of every level: Z^l_b = conv(Y^l_b, folded W_l,b), ZT x ZT tiles.
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
      float* ps = work + g * WF;
      const WtBuf Yb = pl.lev[l];
      const int Hl = pl.Hs[l], Wl = pl.Ws[l];
      if (Hl <= 2 && Wl <= 2) {  // the whole band is this item (at most 16 products)
        const WtBuf Zb = pl.zb[l];
        tiny_band_conv<K>(ps + Yb.off + b * Yb.band + Yb.prow * Yb.stride + Yb.pcol, Yb.stride,
                          wsm + (1 + 4 * (l - 1) + b) * wb, ps + Zb.off + b * Zb.band, Zb.stride, Hl, Wl);
        continue;
      }
      float z[ZT][ZT];
#pragma unroll
      for (int o = 0; o < ZT; ++o)
#pragma unroll
        for (int j = 0; j < ZT; ++j) z[o][j] = 0.f;
      conv_tile<K, ZT, ZT>(ps + Yb.off + b * Yb.band + p0 * Yb.stride + q0, Yb.stride,
                           wsm + (1 + 4 * (l - 1) + b) * wb, z);
      const WtBuf Zb = pl.zb[l];
      float* dst = ps + Zb.off + b * Zb.band + p0 * Zb.stride + q0;
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

    // (2) final tiles: base convolution + synthesis + store.
    if (pl.ftp == WT_TP) final_tiles<K, T, WT_TP>(pl, work, xs, wsm, bias, y, n0, c, np, tid, 0, 0, 0, pl.H, pl.W);
    else final_tiles<K, T, WT_TP / 2>(pl, work, xs, wsm, bias, y, n0, c, np, tid, 0, 0, 0, pl.H, pl.W);
    if (ASYNC && !tma && dbl) cp_async_wait_all();  // this thread's copies of the next unit have landed
    __syncthreads();                 // ... and all reads of unit u are done
  }  // unit loop
}

template <int K, typename T, bool ROT>
static cudaError_t launch_fwd_t(const WtFwdPlan& pl, const CUtensorMap& tmx, const void* x, const float* w_base,
                                const float* b_base, const float* w_sub, const float* s_base,
                                const float* s_w, void* y, cudaStream_t stream) {
  auto kern = fwd_kernel<K, T, ROT>;
  cudaError_t e = ensure_smem((const void*)kern, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  const int per_sm = occupancy((const void*)kern, WT_FWD_THREADS, pl.smem_bytes);
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const long long units = (long long)pl.C * pl.groups;
  long long slots = (long long)(per_sm < 1 ? 1 : per_sm) * sms;
  const unsigned grid = (unsigned)(units < slots ? units : slots);
  kern<<<grid, WT_FWD_THREADS, pl.smem_bytes, stream>>>(pl, tmx, static_cast<const T*>(x), w_base, b_base,
                                                        w_sub, s_base, s_w, static_cast<T*>(y));
  return cudaGetLastError();
}

template <typename T, bool ROT>
static cudaError_t launch_fwd_k(const WtFwdPlan& pl, const CUtensorMap& tmx, const void* x,
                                const float* w_base, const float* b_base, const float* w_sub,
                                const float* s_base, const float* s_w, void* y, cudaStream_t stream) {
  switch (pl.K) {
    case 3: return launch_fwd_t<3, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 5: return launch_fwd_t<5, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 7: return launch_fwd_t<7, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 9: return launch_fwd_t<9, T, ROT>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd(const WtFwdPlan& pl, const CUtensorMap& tmx, int dtype, bool rotate, const void* x,
                       const float* w_base, const float* b_base, const float* w_sub, const float* s_base,
                       const float* s_w, void* y, cudaStream_t stream) {
  if (dtype == 0)
    return rotate ? launch_fwd_k<float, true>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_fwd_k<float, false>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  if (dtype == 1)
    return rotate ? launch_fwd_k<__half, true>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_fwd_k<__half, false>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  return rotate ? launch_fwd_k<__nv_bfloat16, true>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                : launch_fwd_k<__nv_bfloat16, false>(pl, tmx, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
}

template <typename T>
static const void* fwd_pick(int k) {
  switch (k) {
    case 3: return (const void*)fwd_kernel<3, T, false>;
    case 5: return (const void*)fwd_kernel<5, T, false>;
    case 7: return (const void*)fwd_kernel<7, T, false>;
    case 9: return (const void*)fwd_kernel<9, T, false>;
    default: return nullptr;
  }
}

int fwd_regs(int k, int dtype) {
  static std::mutex mu;
  static int cache[4][3];  // k = 3, 5, 7, 9; dtype; 0 = not yet read
  const int ki = (k - 3) / 2;
  if (ki < 0 || ki > 3 || dtype < 0 || dtype > 2) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[ki][dtype] == 0) {
    const void* f = dtype == 0 ? fwd_pick<float>(k) : dtype == 1 ? fwd_pick<__half>(k) : fwd_pick<__nv_bfloat16>(k);
    cudaFuncAttributes a;
    if (!f || cudaFuncGetAttributes(&a, f) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[ki][dtype] = a.numRegs;
  }
  return cache[ki][dtype];
}

unsigned int take_fwd_faults() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_faults, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_fwd_faults, &z, sizeof(z));
  return v;
}

}  // namespace wt
