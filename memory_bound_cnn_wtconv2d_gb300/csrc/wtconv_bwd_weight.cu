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
// One CTA owns channel c and a chunk of the batch.  Planes of x and dy are
// read once into shared memory, both pyramids are rebuilt there
// (unnormalised, so G_l is recovered as 4^-l times the sum), and every
// thread accumulates the K*K correlations of its fixed 4x4 tiles in
// registers across the chunk.  At the end the tile sums of each band are
// reduced through shared memory into one record per (chunk, channel); a
// second kernel adds the records of all chunks in a fixed order, so the
// result does not depend on scheduling.
#include "wtconv_device.cuh"
#include "wtconv_launch.h"

namespace wt {

// Bounded waits that gave up (see mbar_wait_bounded); read by take_bw_faults().
static __device__ unsigned int g_bw_faults;

// TR = 8: 8x4 tiles, one per thread; TR = 4: 4x4 tiles, up to two per thread.
// Tiles are 4 columns wide so neighbouring lanes read neighbouring 16-byte
// chunks of a row (no shared-memory bank conflicts within a row).
template <int K, typename T, int TR>
__global__ void __launch_bounds__(WT_BW_THREADS)
    bw_kernel(const __grid_constant__ WtBwPlan pl, const __grid_constant__ CUtensorMap tmx,
              const __grid_constant__ CUtensorMap tmd, const T* __restrict__ x, const T* __restrict__ dy,
              float* __restrict__ part) {
  extern __shared__ __align__(16) float sm_raw[];
  float* const sm = align_smem128(sm_raw);  // TMA box destinations need 128-byte alignment
  constexpr int KK = K * K;
  constexpr int NT = WT_BW_THREADS;
  constexpr int MI = TR == 8 ? 1 : WT_BW_MAX_ITEMS;
  constexpr int TC = 4;
  constexpr bool ASYNC = sizeof(T) == 4;
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L;
  const int c = blockIdx.x % C;
  const int gi = blockIdx.x / C;
  const int n_begin = gi * pl.chunk;
  const int n_end = min(pl.N, n_begin + pl.chunk);
  constexpr int R = K / 2;
  const int XBF = pl.xbf, DBF = pl.dbf, WF = pl.wf;
  const int ipp = pl.items_per_plane;
  float* const work = sm + pl.work_off;
  const float* const xf = reinterpret_cast<const float*>(x);
  const float* const dyf = reinterpret_cast<const float*>(dy);
  // TMA path (float32, 16-byte rows): one thread issues the x and dy box
  // copies of a batch into input slot `slot`; both complete on mbar[slot].
  const bool tma = ASYNC && pl.use_tma;
  uint64_t* const mbar = reinterpret_cast<uint64_t*>(sm + pl.mb_off);
  __shared__ int s_ok;
  uint32_t parity = 0;  // thread 0: phase parity of mbar[0] (bit 0) and mbar[1] (bit 1)
  auto issue = [&](int n0, int s) {
    float* const dst = sm + s * pl.islot;
    fence_proxy_async();  // earlier generic accesses of the set precede the copies
    mbar_arrive_expect_tx(&mbar[s], pl.tma_bytes);
    tma_load_4d(dst, &tmx, -4, -R, c, n0, &mbar[s]);
    tma_load_4d(dst + pl.xr, &tmd, 0, 0, c, n0, &mbar[s]);
  };

  // Zeroed once: interiors are rewritten per batch, margins stay zero (the
  // box copies write whole padded planes themselves).
  if (tma) zero_smem(work, pl.P * WF, tid, NT);
  else zero_smem(sm, pl.work_off + pl.P * WF, tid, NT);

  float acc[MI][KK];
  float gs[MI];
#pragma unroll
  for (int s = 0; s < MI; ++s) {
    gs[s] = 0.f;
#pragma unroll
    for (int t = 0; t < KK; ++t) acc[s][t] = 0.f;
  }
  if (tma && tid == 0) {
    mbar_init(&mbar[0], 1);
    mbar_init(&mbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();

  if (tma) {
    if (tid == 0 && n_begin < n_end) issue(n_begin, 0);
  } else if (ASYNC && n_begin < n_end) {  // first batch
    const int np0 = min(pl.P, n_end - n_begin);
    load_planes_async(sm, XBF, pl.xs[0], xf, n_begin, np0, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
    load_planes_async(sm + pl.xr, DBF, pl.ds[0], dyf, n_begin, np0, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
    cp_async_commit();
    cp_async_wait_all();
  }
  int slot = 0;
  for (int nb = n_begin; nb < n_end; nb += pl.P, slot ^= 1) {
    const int np = min(pl.P, n_end - nb);
    float* const in_x = sm + slot * pl.islot;  // this batch's raw x planes
    float* const in_d = in_x + pl.xr;          // ... and raw dy planes
    if (tma) {
      if (tid == 0) {
        const bool ok = mbar_wait_bounded(&mbar[slot], (parity >> slot) & 1u);
        parity ^= 1u << slot;
        if (ok && nb + pl.P < n_end) issue(nb + pl.P, slot ^ 1);  // the other set was last read by batch nb-P
        s_ok = ok;
      }
    } else if (!ASYNC) {
      load_planes<T>(in_x, XBF, pl.xs[0], x, nb, np, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
      load_planes<T>(in_d, DBF, pl.ds[0], dy, nb, np, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
    } else if (nb + pl.P < n_end) {  // prefetch the next batch into the other slot
      const int n1 = nb + pl.P, np1 = min(pl.P, n_end - n1);
      float* const nxt = sm + (slot ^ 1) * pl.islot;
      load_planes_async(nxt, XBF, pl.xs[0], xf, n1, np1, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
      load_planes_async(nxt + pl.xr, DBF, pl.ds[0], dyf, n1, np1, c, C, pl.H, pl.W, pl.vec_ok != 0, pl.ld_pp, pl.ld_w, tid, NT);
      cp_async_commit();
    }
    __syncthreads();  // this batch's planes are visible
    if (tma && !s_ok) {  // the copy did not complete in time: record it and stop (uniform exit)
      if (tid == 0) {
        atomicAdd(&g_bw_faults, 1u);
        mbar_wait_bounded(&mbar[slot], ((parity >> slot) & 1u) ^ 1u);  // let the copy in flight land
      }
      __syncthreads();
      return;  // partial sums are not written: the caller sees the fault count
    }

    // Both pyramids: levels 1+2 fused, then 3..L.
    if (L == 1) {
      haar_level(in_x, XBF, work, WF, np, pl.xs[0], pl.xs[1], pl.Hs[1], pl.Ws[1], pl.an_pp[1], pl.an_w[1], tid, NT);
      haar_level(in_d, DBF, work, WF, np, pl.ds[0], pl.ds[1], pl.Hs[1], pl.Ws[1], pl.an_pp[1], pl.an_w[1], tid, NT);
    } else {
      haar_levels12(in_x, XBF, work, WF, np, pl.xs[0], pl.xs[1], pl.xs[2], pl.Hs[1], pl.Ws[1], pl.Hs[2], pl.Ws[2],
                    pl.an_pp[2], pl.an_w[2], tid, NT);
      haar_levels12(in_d, DBF, work, WF, np, pl.ds[0], pl.ds[1], pl.ds[2], pl.Hs[1], pl.Ws[1], pl.Hs[2], pl.Ws[2],
                    pl.an_pp[2], pl.an_w[2], tid, NT);
    }
    __syncthreads();
    for (int l = 3; l <= L; ++l) {
      haar_level(work, WF, work, WF, np, pl.xs[l - 1], pl.xs[l], pl.Hs[l], pl.Ws[l], pl.an_pp[l], pl.an_w[l], tid, NT);
      haar_level(work, WF, work, WF, np, pl.ds[l - 1], pl.ds[l], pl.Hs[l], pl.Ws[l], pl.an_pp[l], pl.an_w[l], tid, NT);
      __syncthreads();
    }
#pragma unroll
    for (int s = 0; s < MI; ++s) {
      const int item = tid + s * NT;
      if (item < pl.P * ipp) {
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
          float dsum;
          if (l == 0) {  // raw planes; x's interior starts 4 floats into each row
            const float* xw = in_x + g * XBF + Xb.off + p0 * Xb.stride + q0;
            const float* dw = in_d + g * DBF + Db.off + p0 * Db.stride + q0;
            dsum = corr_tile<K, TR, TC, 4 - R>(xw, Xb.stride, dw, Db.stride, acc[s]);
            gs[s] += dsum;
          } else {
            const float* ps = work + g * WF;
            dsum = corr_tile<K, TR, TC>(ps + Xb.off + b * Xb.band + p0 * Xb.stride + q0, Xb.stride,
                                        ps + Db.off + b * Db.band + p0 * Db.stride + q0, Db.stride, acc[s]);
          }
        }
      }
    }
    if (ASYNC && !tma) cp_async_wait_all();  // this thread's copies of the next batch have landed
    __syncthreads();                         // ... and every read of this batch is done
  }

  // Tile sums -> shared memory -> one record per band.
  float* red = sm;
  const int rs = KK + 1;
#pragma unroll
  for (int s = 0; s < MI; ++s) {
    const int item = tid + s * NT;
    if (item < pl.P * ipp) {
#pragma unroll
      for (int t = 0; t < KK; ++t) red[item * rs + t] = acc[s][t];
      red[item * rs + KK] = gs[s];
    }
  }
  __syncthreads();
  float* rec = part + ((size_t)gi * C + c) * pl.part_stride;
  for (int qd = tid; qd < pl.nbands * rs; qd += NT) {
    const int B = qd / rs;
    const int t = qd - B * rs;
    const int l = (B == 0) ? 0 : 1 + ((B - 1) >> 2);
    const int b = (B == 0) ? 0 : ((B - 1) & 3);
    const int tiles = pl.tr[l] * pl.tc[l];
    const int first = pl.item_begin[l] + b * tiles;
    float sum = 0.f;
    if (B == 0 || t < KK) {
      for (int g = 0; g < pl.P; ++g)
        for (int i = 0; i < tiles; ++i) sum += red[(g * ipp + first + i) * rs + t];
    }
    rec[qd] = sum;
  }
}

// Adds the records of all chunks of channel c in chunk order and unfolds the
// scales.  One warp per (channel, band): lane t owns taps t, t+32, t+64; the
// scale gradient <W, G> is reduced with a fixed shuffle tree, so the result
// does not depend on scheduling.
__global__ void bw_finalize_kernel(const __grid_constant__ WtBwPlan pl, const float* __restrict__ part,
                                   const float* __restrict__ w_base, const float* __restrict__ b_base,
                                   const float* __restrict__ w_sub, const float* __restrict__ s_base,
                                   const float* __restrict__ s_w, float* __restrict__ dw_base,
                                   float* __restrict__ db_base, float* __restrict__ dw_sub,
                                   float* __restrict__ ds_base, float* __restrict__ ds_w) {
  const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int C = pl.C, K = pl.K, KK = K * K, rs = KK + 1;
  if (warp >= C * pl.nbands) return;  // whole warps exit together
  const int c = warp / pl.nbands;
  const int B = warp - c * pl.nbands;
  const float* rec = part + (size_t)c * pl.part_stride + (size_t)B * rs;
  const size_t gstride = (size_t)C * pl.part_stride;
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
  float dot = 0.f;
  for (int t = lane; t < KK; t += 32) {
    float G = 0.f;
    for (int g = 0; g < pl.groups; ++g) G += rec[g * gstride + t];
    G = ldexpf(G, -2 * l);  // level-l sums were taken on unnormalised coefficients
    dw[t] = scale * G;
    dot = fmaf(w[t], G, dot);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (lane == 0) {
    if (B == 0) {
      float gsum = 0.f;
      for (int g = 0; g < pl.groups; ++g) gsum += rec[g * gstride + KK];
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
  auto kern = pl.tbr == 8 ? bw_kernel<K, T, 8> : bw_kernel<K, T, 4>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)pl.C * (unsigned)pl.groups;
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
  const int warps = pl.C * pl.nbands;
  const int threads = 256;
  bw_finalize_kernel<<<(warps * 32 + threads - 1) / threads, threads, 0, stream>>>(
      pl, part, w_base, b_base, w_sub, s_base, s_w, dw_base, db_base, dw_sub, ds_base, ds_w);
  return cudaGetLastError();
}

unsigned int take_bw_faults() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_bw_faults, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_bw_faults, &z, sizeof(z));
  return v;
}

}  // namespace wt
