// Fused WTConv2d forward pass and input-gradient pass (sm_103a).
//
// One CTA owns P planes of one channel.  The planes cross HBM once: they are
// read into shared memory, the Haar pyramid is rebuilt there, every level is
// convolved with scale-folded weights, and the synthesis of all levels is
// summed tile by tile from the coarsest level down, so that the finest tiles
// write the output straight from registers.
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
// Here (2) is evaluated in shared memory from level L to 2 as running sums
// T^{l-1}[2p+u][2q+v] = sum_b sign_b(u,v) Z^l_b[p][q] + T^l[p][q] (the same
// sum, grouped by coarse pixel), and level 1 adds it in registers.  The
// 2^-l normalisations of analysis and synthesis (4^-l in total) are folded
// into the level-l weights, so the butterflies are pure adds.
//
// The input-gradient pass is the same kernel with every kernel rotated by
// 180 degrees and no bias: the layer map is A = s_b*Conv_b + sum_l F_l^T K_l F_l
// with orthonormal F_l, so A^T = s_b*Conv_b^T + sum_l F_l^T K_l^T F_l and the
// transpose of a same-padded odd-k correlation is the correlation with the
// rotated kernel.
#include "wtconv_device.cuh"
#include "wtconv_launch.h"

namespace wt {

// v[2o+u][2j+v] += sign_b(u, v) * z[o][j] for one band b.
template <int TP, int TQ>
__device__ __forceinline__ void add_band(float (&v)[2 * TP][2 * TQ], const float (&z)[TP][TQ], int b) {
#pragma unroll
  for (int o = 0; o < TP; ++o)
#pragma unroll
    for (int j = 0; j < TQ; ++j) {
      const float zz = z[o][j];
      v[2 * o][2 * j] += zz;
      v[2 * o][2 * j + 1] += (b & 2) ? -zz : zz;             // sign (-1)^v for bands 2, 3
      v[2 * o + 1][2 * j] += (b & 1) ? -zz : zz;             // sign (-1)^u for bands 1, 3
      v[2 * o + 1][2 * j + 1] += (b == 1 || b == 2) ? -zz : zz;
    }
}

template <int K, typename T, bool ROT>
__global__ void __launch_bounds__(WT_FWD_THREADS)
    fwd_kernel(const __grid_constant__ WtFwdPlan pl, const T* __restrict__ x,
               const float* __restrict__ w_base, const float* __restrict__ b_base,
               const float* __restrict__ w_sub, const float* __restrict__ s_base,
               const float* __restrict__ s_w, T* __restrict__ y) {
  extern __shared__ __align__(16) float sm[];
  constexpr int KK = K * K;
  constexpr int NT = WT_FWD_THREADS;
  constexpr int TP = WT_TP, TQ = WT_TQ;
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L;
  const int c = blockIdx.x % C;
  const int n0 = (blockIdx.x / C) * pl.P;
  const int np = min(pl.P, pl.N - n0);
  const int PF = pl.plane_floats;

  zero_smem(sm, pl.P * PF, tid, NT);

  // (3) fold scales: base kernel * s_base; level-l kernels * s_w * 4^-l.
  float* wsm = sm + pl.w_off;
  const int wb = pl.w_band;
  for (int i = tid; i < (1 + 4 * L) * wb; i += NT) {
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
        v = ldexpf(s_w[ch], -2 * (l + 1)) * w_sub[(size_t)ch * KK + ts];
      }
    }
    wsm[i] = v;
  }
  const float bias = (!ROT && b_base != nullptr) ? s_base[c] * b_base[c] : 0.f;
  __syncthreads();

  load_planes<T>(sm, PF, pl.lev[0], x, n0, np, c, C, pl.H, pl.W, pl.vec_ok != 0, tid, NT);
  __syncthreads();

  // (1) Haar pyramid, levels 1..L, on chip.
  for (int l = 1; l <= L; ++l) {
    haar_level(sm, PF, np, pl.lev[l - 1], pl.lev[l], pl.Hs[l], pl.Ws[l], tid, NT);
    __syncthreads();
  }

  // (2) synthesis, coarse levels L..2 -> running sums T^{l-1}.
  for (int l = L; l >= 2; --l) {
    const WtBuf Yb = pl.lev[l];
    const WtBuf Ti = pl.syn[l];      // read (l < L)
    const WtBuf To = pl.syn[l - 1];  // write
    const int tcn = pl.tc[l];
    const int per_plane = pl.tr[l] * tcn;
    const int Hd = pl.Hs[l - 1], Wd = pl.Ws[l - 1];
    const float* wl = wsm + (1 + 4 * (l - 1)) * wb;
    for (int it = tid; it < np * per_plane; it += NT) {
      const int g = it / per_plane;
      const int rem = it - g * per_plane;
      const int tp = rem / tcn;
      const int p0 = tp * TP, q0 = (rem - tp * tcn) * TQ;
      float* ps = sm + g * PF;
      float v[2 * TP][2 * TQ];
#pragma unroll
      for (int o = 0; o < TP; ++o) {
        float tv[TQ];
        if (l < L) {
          lds_row<TQ / 4>(ps + Ti.off + (p0 + o) * Ti.stride + q0, tv);
        } else {
#pragma unroll
          for (int j = 0; j < TQ; ++j) tv[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < TQ; ++j) {
          v[2 * o][2 * j] = tv[j];
          v[2 * o][2 * j + 1] = tv[j];
          v[2 * o + 1][2 * j] = tv[j];
          v[2 * o + 1][2 * j + 1] = tv[j];
        }
      }
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float z[TP][TQ];
#pragma unroll
        for (int o = 0; o < TP; ++o)
#pragma unroll
          for (int j = 0; j < TQ; ++j) z[o][j] = 0.f;
        conv_tile<K, TP, TQ>(ps + Yb.off + b * Yb.band + p0 * Yb.stride + q0, Yb.stride, wl + b * wb, z);
        add_band<TP, TQ>(v, z, b);
      }
#pragma unroll
      for (int oo = 0; oo < 2 * TP; ++oo) {
        const int i = 2 * p0 + oo;
        if (i < Hd) {
          float* dst = ps + To.off + i * To.stride;
#pragma unroll
          for (int jj = 0; jj < 2 * TQ; ++jj)
            if (2 * q0 + jj < Wd) dst[2 * q0 + jj] = v[oo][jj];
        }
      }
    }
    __syncthreads();
  }

  // Level 1 + base conv: outputs straight from registers.
  {
    const WtBuf X = pl.lev[0];
    const WtBuf Y1 = pl.lev[1];
    const WtBuf T1 = pl.syn[1];
    const int tcn = pl.tc[1];
    const int per_plane = pl.tr[1] * tcn;
    const int H = pl.H, W = pl.W;
    const size_t HW = (size_t)H * W;
    const float* w1 = wsm + wb;
    for (int it = tid; it < np * per_plane; it += NT) {
      const int g = it / per_plane;
      const int rem = it - g * per_plane;
      const int tp = rem / tcn;
      const int p0 = tp * TP, q0 = (rem - tp * tcn) * TQ;
      const float* ps = sm + g * PF;
      float v[2 * TP][2 * TQ];
#pragma unroll
      for (int o = 0; o < TP; ++o) {
        float tv[TQ];
        if (L > 1) {
          lds_row<TQ / 4>(ps + T1.off + (p0 + o) * T1.stride + q0, tv);
        } else {
#pragma unroll
          for (int j = 0; j < TQ; ++j) tv[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < TQ; ++j) {
          v[2 * o][2 * j] = tv[j] + bias;
          v[2 * o][2 * j + 1] = tv[j] + bias;
          v[2 * o + 1][2 * j] = tv[j] + bias;
          v[2 * o + 1][2 * j + 1] = tv[j] + bias;
        }
      }
      conv_tile<K, 2 * TP, 2 * TQ>(ps + X.off + 2 * p0 * X.stride + 2 * q0, X.stride, wsm, v);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float z[TP][TQ];
#pragma unroll
        for (int o = 0; o < TP; ++o)
#pragma unroll
          for (int j = 0; j < TQ; ++j) z[o][j] = 0.f;
        conv_tile<K, TP, TQ>(ps + Y1.off + b * Y1.band + p0 * Y1.stride + q0, Y1.stride, w1 + b * wb, z);
        add_band<TP, TQ>(v, z, b);
      }
      T* plane = y + ((size_t)(n0 + g) * C + c) * HW;
      const int j0 = 2 * q0;
      constexpr int V = Vec16<T>::N;
      const bool full_row = pl.vec_ok && (j0 + 2 * TQ <= W);
#pragma unroll
      for (int oo = 0; oo < 2 * TP; ++oo) {
        const int i = 2 * p0 + oo;
        if (i < H) {
          T* dst = plane + (size_t)i * W + j0;
          if (full_row) {
#pragma unroll
            for (int s = 0; s < 2 * TQ; s += V) stg16<T>(dst + s, &v[oo][s]);
          } else {
#pragma unroll
            for (int jj = 0; jj < 2 * TQ; ++jj)
              if (j0 + jj < W) dst[jj] = from_f32<T>(v[oo][jj]);
          }
        }
      }
    }
  }
}

template <int K, typename T, bool ROT>
static cudaError_t launch_fwd_t(const WtFwdPlan& pl, const void* x, const float* w_base,
                                const float* b_base, const float* w_sub, const float* s_base,
                                const float* s_w, void* y, cudaStream_t stream) {
  auto kern = fwd_kernel<K, T, ROT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)pl.C * (unsigned)pl.groups;
  kern<<<grid, WT_FWD_THREADS, pl.smem_bytes, stream>>>(pl, static_cast<const T*>(x), w_base, b_base,
                                                        w_sub, s_base, s_w, static_cast<T*>(y));
  return cudaGetLastError();
}

template <typename T, bool ROT>
static cudaError_t launch_fwd_k(const WtFwdPlan& pl, const void* x, const float* w_base,
                                const float* b_base, const float* w_sub, const float* s_base,
                                const float* s_w, void* y, cudaStream_t stream) {
  switch (pl.K) {
    case 3: return launch_fwd_t<3, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 5: return launch_fwd_t<5, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 7: return launch_fwd_t<7, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 9: return launch_fwd_t<9, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd(const WtFwdPlan& pl, int dtype, bool rotate, const void* x, const float* w_base,
                       const float* b_base, const float* w_sub, const float* s_base, const float* s_w,
                       void* y, cudaStream_t stream) {
  if (dtype == 0)
    return rotate ? launch_fwd_k<float, true>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_fwd_k<float, false>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  if (dtype == 1)
    return rotate ? launch_fwd_k<__half, true>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_fwd_k<__half, false>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  return rotate ? launch_fwd_k<__nv_bfloat16, true>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                : launch_fwd_k<__nv_bfloat16, false>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
}

}  // namespace wt
