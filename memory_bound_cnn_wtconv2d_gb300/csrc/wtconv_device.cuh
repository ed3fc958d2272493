// Device building blocks of libwtconv (sm_103a).
//
// Depthwise convolution and Haar butterflies are not dense contractions, so
// everything here runs on the FP32 pipes: tiles of outputs per thread with
// register-resident weights and sliding rows read from shared memory with
// 16-byte loads.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "wtconv_plan.h"

namespace wt {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ int fdiv(int n, const WtDiv& f) {
  return (int)((__umulhi((uint32_t)n, f.mul) + (uint32_t)n) >> f.shift);
}

// Elements per 16-byte global access.
template <typename T> struct Vec16 { static constexpr int N = 16 / (int)sizeof(T); };

// 16-byte global load of 16/sizeof(T) elements, widened to float.
template <typename T>
__device__ __forceinline__ void ldg16(const T* __restrict__ p, float (&v)[Vec16<T>::N]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  if constexpr (sizeof(T) == 4) {
    v[0] = __uint_as_float(u.x);
    v[1] = __uint_as_float(u.y);
    v[2] = __uint_as_float(u.z);
    v[3] = __uint_as_float(u.w);
  } else {
    const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = to_f32(h[e]);
  }
}

// 16-byte global store of 16/sizeof(T) floats, rounded to T (nearest even).
template <typename T>
__device__ __forceinline__ void stg16(T* __restrict__ p, const float* v) {
  uint4 u;
  if constexpr (sizeof(T) == 4) {
    u.x = __float_as_uint(v[0]);
    u.y = __float_as_uint(v[1]);
    u.z = __float_as_uint(v[2]);
    u.w = __float_as_uint(v[3]);
  } else {
    T* h = reinterpret_cast<T*>(&u);
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = from_f32<T>(v[e]);
  }
  *reinterpret_cast<uint4*>(p) = u;
}

// Stores N consecutive outputs (rounded to T) with one N*sizeof(T)-byte
// access when that is 8 or 16 bytes; dst must be aligned to that size.
template <typename T, int N>
__device__ __forceinline__ void stg_row(T* __restrict__ dst, const float* v) {
  constexpr int BYTES = N * (int)sizeof(T);
  if constexpr (BYTES == 16) {
    stg16<T>(dst, v);
  } else if constexpr (BYTES == 8) {
    uint2 u;
    T* h = reinterpret_cast<T*>(&u);
#pragma unroll
    for (int e = 0; e < N; ++e) h[e] = from_f32<T>(v[e]);
    *reinterpret_cast<uint2*>(dst) = u;
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) dst[e] = from_f32<T>(v[e]);
  }
}

// NV aligned float4 loads from shared memory.
template <int NV>
__device__ __forceinline__ void lds_row(const float* p, float (&seg)[4 * NV]) {
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const float4 t = *reinterpret_cast<const float4*>(p + 4 * v);
    seg[4 * v + 0] = t.x;
    seg[4 * v + 1] = t.y;
    seg[4 * v + 2] = t.z;
    seg[4 * v + 3] = t.w;
  }
}

// K*K weights (stored with a stride rounded up to 4 floats, 16-byte aligned).
template <int K>
__device__ __forceinline__ void load_weights(const float* w, float (&wr)[K * K]) {
  constexpr int KK = K * K;
#pragma unroll
  for (int t = 0; t < KK; t += 4) {
    const float4 q = *reinterpret_cast<const float4*>(w + t);
    wr[t] = q.x;
    if (t + 1 < KK) wr[t + 1] = q.y;
    if (t + 2 < KK) wr[t + 2] = q.z;
    if (t + 3 < KK) wr[t + 3] = q.w;
  }
}

// acc[o][j] += sum_{du,dv} w[du][dv] * win[(o+du)*stride + j+dv]
// `win` is the top-left corner of the (TR+K-1) x (TC+K-1) input window,
// 16-byte aligned; rows are read as whole float4s (the buffer's row stride
// leaves room for the over-read).
template <int K, int TR, int TC>
__device__ __forceinline__ void conv_tile(const float* __restrict__ win, int stride,
                                          const float* __restrict__ w, float (&acc)[TR][TC]) {
  constexpr int NV = (TC + K - 1 + 3) / 4;
  float wr[K * K];
  load_weights<K>(w, wr);
#pragma unroll
  for (int a = 0; a < TR + K - 1; ++a) {
    float seg[4 * NV];
    lds_row<NV>(win + a * stride, seg);
#pragma unroll
    for (int o = 0; o < TR; ++o) {
      const int du = a - o;
      if (du >= 0 && du < K) {
#pragma unroll
        for (int dv = 0; dv < K; ++dv)
#pragma unroll
          for (int j = 0; j < TC; ++j) acc[o][j] = fmaf(wr[du * K + dv], seg[j + dv], acc[o][j]);
      }
    }
  }
}

// seg[0..N) = p[OFF .. OFF+N) with the widest aligned shared loads; p is
// 16-byte aligned and OFF, N are compile-time, so the pattern unrolls fully.
template <int OFF, int N, int I = 0>
__device__ __forceinline__ void lds_span(const float* p, float (&seg)[N]) {
  if constexpr (I < N) {
    constexpr int a = OFF + I;
    if constexpr (a % 4 == 0 && I + 4 <= N) {
      const float4 t = *reinterpret_cast<const float4*>(p + a);
      seg[I] = t.x; seg[I + 1] = t.y; seg[I + 2] = t.z; seg[I + 3] = t.w;
      lds_span<OFF, N, I + 4>(p, seg);
    } else if constexpr (a % 2 == 0 && I + 2 <= N) {
      const float2 t = *reinterpret_cast<const float2*>(p + a);
      seg[I] = t.x; seg[I + 1] = t.y;
      lds_span<OFF, N, I + 2>(p, seg);
    } else {
      seg[I] = p[a];
      lds_span<OFF, N, I + 1>(p, seg);
    }
  }
}

// conv_tile for a window whose first column sits OFF floats after a 16-byte
// boundary: reads exactly TC+K-1 floats per row.
template <int K, int TR, int TC, int OFF>
__device__ __forceinline__ void conv_tile_off(const float* __restrict__ row0, int stride,
                                              const float* __restrict__ w, float (&acc)[TR][TC]) {
  float wr[K * K];
  load_weights<K>(w, wr);
#pragma unroll
  for (int a = 0; a < TR + K - 1; ++a) {
    float seg[TC + K - 1];
    lds_span<OFF, TC + K - 1>(row0 + a * stride, seg);
#pragma unroll
    for (int o = 0; o < TR; ++o) {
      const int du = a - o;
      if (du >= 0 && du < K) {
#pragma unroll
        for (int dv = 0; dv < K; ++dv)
#pragma unroll
          for (int j = 0; j < TC; ++j) acc[o][j] = fmaf(wr[du * K + dv], seg[j + dv], acc[o][j]);
      }
    }
  }
}

// acc[du*K+dv] += sum_{o,j} d[o][j] * win[(o+du)*stride + j+dv]   (weight-gradient correlation)
// Returns the sum of the d tile (for the bias gradient).
// The window's first column sits OFF floats after the 16-byte-aligned `win`
// (OFF = 0: whole float4s are read, the row stride leaves room; else exactly
// TC+K-1 floats are read).
template <int K, int TR, int TC, int OFF = 0>
__device__ __forceinline__ float corr_tile(const float* __restrict__ win, int wstride,
                                           const float* __restrict__ dsrc, int dstride,
                                           float (&acc)[K * K]) {
  constexpr int NV = (TC + K - 1 + 3) / 4;
  constexpr int NS = OFF == 0 ? 4 * NV : TC + K - 1;
  static_assert(TC % 4 == 0, "tile width must be a multiple of 4");
  float d[TR][TC];
  float dsum = 0.f;
#pragma unroll
  for (int o = 0; o < TR; ++o) {
    float row[TC];
    lds_row<TC / 4>(dsrc + o * dstride, row);
#pragma unroll
    for (int j = 0; j < TC; ++j) {
      d[o][j] = row[j];
      dsum += row[j];
    }
  }
#pragma unroll
  for (int a = 0; a < TR + K - 1; ++a) {
    float seg[NS];
    if constexpr (OFF == 0) lds_row<NV>(win + a * wstride, seg);
    else lds_span<OFF, NS>(win + a * wstride, seg);
#pragma unroll
    for (int o = 0; o < TR; ++o) {
      const int du = a - o;
      if (du >= 0 && du < K) {
#pragma unroll
        for (int dv = 0; dv < K; ++dv)
#pragma unroll
          for (int j = 0; j < TC; ++j) acc[du * K + dv] = fmaf(d[o][j], seg[j + dv], acc[du * K + dv]);
      }
    }
  }
  return dsum;
}

// Bands of at most 2 x 2 coefficients (the deep levels of small planes,
// whose ceil-halved sizes end at 1 x 1): a k x k kernel on such a band only
// ever meets the band's own <= 4 coefficients, so the convolution and the
// correlation are at most 16 products, written out here instead of a whole
// coefficient tile.  `y`, `x` and `d` point at the band's interior origin;
// the band buffers keep zero margins around the interior, so the 2 x 2 block
// read here is the band itself, zero-extended.
//   z[p][q] = sum_{i,j} w[(i-p+r)*K + (j-q+r)] * y[i][j]            (p < Hl, q < Wl)
template <int K>
__device__ __forceinline__ void tiny_band_conv(const float* __restrict__ y, int ys, const float* __restrict__ w,
                                               float* __restrict__ z, int zs, int Hl, int Wl) {
  constexpr int R = K / 2;
  const float v[2][2] = {{y[0], y[1]}, {y[ys], y[ys + 1]}};
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (p < Hl && q < Wl) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int j = 0; j < 2; ++j) acc = fmaf(w[(i - p + R) * K + (j - q + R)], v[i][j], acc);
        z[p * zs + q] = acc;
      }
    }
}

//   acc[du*K+dv] += sum_{p,q} x[p+du-r][q+dv-r] * d[p][q]: every product of
//   one of the band's x coefficients with one of its d coefficients lands on
//   exactly one tap, so 16 products cover the whole correlation.
template <int K>
__device__ __forceinline__ void tiny_band_corr(const float* __restrict__ x, int xs, const float* __restrict__ d,
                                               int ds, float (&acc)[K * K]) {
  constexpr int R = K / 2;
  const float xv[2][2] = {{x[0], x[1]}, {x[xs], x[xs + 1]}};
  const float dv[2][2] = {{d[0], d[1]}, {d[ds], d[ds + 1]}};
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float& a = acc[(i - p + R) * K + (j - q + R)];
          a = fmaf(xv[i][j], dv[p][q], a);
        }
}

// One Haar analysis level on the planes g < np of a CTA:
//   dst_b[p][q] = sum_{u,v} sign_b(u,v) * src[2p+u][2q+v],  p < Hl, q < Wl
// (unnormalised: the 1/2 per level is folded into the weights).  Reads past
// the source interior hit its zero margin.  Plane g's source buffer starts at
// sbase + g*sps, its destination at dbase + g*dps.
__device__ __forceinline__ void haar_level(const float* sbase, int sps, float* dbase, int dps, int np,
                                           const WtBuf S, const WtBuf D, int Hl, int Wl, const WtDiv& dpp,
                                           const WtDiv& dw, int tid, int nthreads) {
  const int per_plane = Hl * Wl;
  for (int it = tid; it < np * per_plane; it += nthreads) {
    const int g = fdiv(it, dpp);
    const int rem = it - g * per_plane;
    const int p = fdiv(rem, dw);
    const int q = rem - p * Wl;
    const float* s = sbase + g * sps + S.off + (2 * p + S.prow) * S.stride + 2 * q + S.pcol;
    const float a = s[0], b = s[1], c = s[S.stride], d = s[S.stride + 1];
    const float s0 = a + b, d0 = a - b, s1 = c + d, d1 = c - d;
    float* o = dbase + g * dps + D.off + (p + D.prow) * D.stride + q + D.pcol;
    o[0] = s0 + s1;           // low-pass
    o[D.band] = s0 - s1;      // row-high:    sign (-1)^u
    o[2 * D.band] = d0 + d1;  // column-high: sign (-1)^v
    o[3 * D.band] = d0 - d1;  // diagonal:    sign (-1)^(u+v)
  }
}

// Unnormalised 2x2 Haar butterfly of (a b / c d): LL, row-high, column-high, diagonal.
__device__ __forceinline__ void butterfly4(float a, float b, float c, float d, float (&o)[4]) {
  const float s0 = a + b, d0 = a - b, s1 = c + d, d1 = c - d;
  o[0] = s0 + s1;
  o[1] = s0 - s1;
  o[2] = d0 + d1;
  o[3] = d0 - d1;
}

// Loads the 4x4 input block at level-2 position (P, Q) of source buffer S.
__device__ __forceinline__ void load_block4(const float* s, const WtBuf S, float (&x)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const float* r = s + a * S.stride;
    if ((S.pcol & 3) == 0) {
      const float4 t = *reinterpret_cast<const float4*>(r);
      x[a][0] = t.x; x[a][1] = t.y; x[a][2] = t.z; x[a][3] = t.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[a][e] = r[e];
    }
  }
}

// Levels 1 and 2 of one 4x4 block (butterflies of haar_levels12) stored at
// level-2 position (P, Q) of the destination buffers D1, D2 of plane base ps.
__device__ __forceinline__ void store_block12(const float (&x)[4][4], float* ps, const WtBuf D1, const WtBuf D2,
                                              int P, int Q, int H1, int W1) {
  float ll[2][2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    float o[2][4];
#pragma unroll
    for (int v = 0; v < 2; ++v) {
      butterfly4(x[2 * u][2 * v], x[2 * u][2 * v + 1], x[2 * u + 1][2 * v], x[2 * u + 1][2 * v + 1], o[v]);
      ll[u][v] = o[v][0];
    }
    const int p = 2 * P + u, q = 2 * Q;
    if (p < H1) {
      float* d = ps + D1.off + (p + D1.prow) * D1.stride + q + D1.pcol;
      if (q + 1 < W1 && (D1.pcol & 1) == 0) {
#pragma unroll
        for (int b = 0; b < 4; ++b) *reinterpret_cast<float2*>(d + b * D1.band) = make_float2(o[0][b], o[1][b]);
      } else {
#pragma unroll
        for (int v = 0; v < 2; ++v)
          if (q + v < W1) {
#pragma unroll
            for (int b = 0; b < 4; ++b) d[b * D1.band + v] = o[v][b];
          }
      }
    }
  }
  float o2[4];
  butterfly4(ll[0][0], ll[0][1], ll[1][0], ll[1][1], o2);
  float* d = ps + D2.off + (P + D2.prow) * D2.stride + Q + D2.pcol;
#pragma unroll
  for (int b = 0; b < 4; ++b) d[b * D2.band] = o2[b];
}

// Haar levels 1 and 2 in one pass: each item reads a 4x4 block of the input
// plane and writes the 2x2 level-1 positions of all four bands and the one
// level-2 position built from their low-pass values (same unnormalised
// butterflies as haar_level).  Items cover the level-2 grid H2 x W2; level-1
// positions past H1 x W1 are skipped (they lie in the zero margin, and the
// input rows/columns they read there are zero).
__device__ __forceinline__ void haar_levels12(const float* sbase, int sps, float* dbase, int dps, int np,
                                              const WtBuf S, const WtBuf D1, const WtBuf D2, int H1, int W1,
                                              int H2, int W2, const WtDiv& dpp, const WtDiv& dw, int tid,
                                              int nthreads) {
  const int per_plane = H2 * W2;
  for (int it = tid; it < np * per_plane; it += nthreads) {
    const int g = fdiv(it, dpp);
    const int rem = it - g * per_plane;
    const int P = fdiv(rem, dw);
    const int Q = rem - P * W2;
    float x[4][4];
    load_block4(sbase + g * sps + S.off + (4 * P + S.prow) * S.stride + 4 * Q + S.pcol, S, x);
    store_block12(x, dbase + g * dps, D1, D2, P, Q, H1, W1);
  }
}

// Levels 1 and 2 straight from np raw 16-bit planes (H*W elements each,
// consecutive in `src`, as the bulk copies leave them): each 4 x 4 block of
// the level-2 grid is read (zero past the plane), widened, written into the
// float32 interior of buffer S of its plane slot (which the base convolution
// reads later), and its butterflies stored as haar_levels12 stores them.
// The grid's blocks cover each plane (4 ceil(ceil(W/2)/2) = 4 ceil(W/4) >= W,
// so a block's first column is inside it), every interior element is
// written once and the margins stay zero.
template <typename T>
__device__ __forceinline__ void widen_block4(const T* plane, int H, int W, int P, int Q, float* sp, const WtBuf S,
                                             bool vec, float (&x)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = 4 * P + a;
#pragma unroll
    for (int e = 0; e < 4; ++e) x[a][e] = 0.f;
    if (i < H) {
      const T* row = plane + i * W + 4 * Q;
      float* dst = sp + S.off + (i + S.prow) * S.stride + 4 * Q + S.pcol;
      if (vec) {
        const uint2 raw = *reinterpret_cast<const uint2*>(row);
        const T* h = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[a][e] = to_f32(h[e]);
        *reinterpret_cast<float4*>(dst) = make_float4(x[a][0], x[a][1], x[a][2], x[a][3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * Q + e < W) {
            x[a][e] = to_f32(row[e]);
            dst[e] = x[a][e];
          }
      }
    }
  }
}

// widen_block4 for rows of even length that are not whole 4-element groups:
// pairs (4-byte loads, 8-byte stores; a pair past the row is skipped).
template <typename T>
__device__ __forceinline__ void widen_block4_pairs(const T* plane, int H, int W, int P, int Q, float* sp,
                                                   const WtBuf S, float (&x)[4][4]) {
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int i = 4 * P + a;
#pragma unroll
    for (int e = 0; e < 4; ++e) x[a][e] = 0.f;
    if (i < H) {
      const T* row = plane + i * W + 4 * Q;
      float* dst = sp + S.off + (i + S.prow) * S.stride + 4 * Q + S.pcol;
#pragma unroll
      for (int e = 0; e < 4; e += 2)
        if (4 * Q + e < W) {
          const uint32_t raw = *reinterpret_cast<const uint32_t*>(row + e);
          const T* h = reinterpret_cast<const T*>(&raw);
          x[a][e] = to_f32(h[0]);
          x[a][e + 1] = to_f32(h[1]);
          *reinterpret_cast<float2*>(dst + e) = make_float2(x[a][e], x[a][e + 1]);
        }
    }
  }
}

template <typename T>
__device__ __forceinline__ void widen_levels12(const T* src, int H, int W, float* sbase, int sps, const WtBuf S,
                                               float* dbase, int dps, int np, const WtBuf D1, const WtBuf D2,
                                               int H1, int W1, int H2, int W2, const WtDiv& dpp, const WtDiv& dw,
                                               int tid, int nthreads) {
  const int HW = H * W;
  const bool vec = (W & 3) == 0 && (S.pcol & 3) == 0;  // 8-byte loads, 16-byte stores
  const bool pairs = !vec && (W & 1) == 0 && ((S.pcol | S.stride) & 1) == 0;
  const int per_plane = H2 * W2;
  if (pairs) {
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int P = fdiv(rem, dw);
      const int Q = rem - P * W2;
      float x[4][4];
      widen_block4_pairs<T>(src + g * HW, H, W, P, Q, sbase + g * sps, S, x);
      store_block12(x, dbase + g * dps, D1, D2, P, Q, H1, W1);
    }
    return;
  }
  for (int it = tid; it < np * per_plane; it += nthreads) {
    const int g = fdiv(it, dpp);
    const int rem = it - g * per_plane;
    const int P = fdiv(rem, dw);
    const int Q = rem - P * W2;
    float x[4][4];
    widen_block4<T>(src + g * HW, H, W, P, Q, sbase + g * sps, S, vec, x);
    store_block12(x, dbase + g * dps, D1, D2, P, Q, H1, W1);
  }
}

// widen_levels12 for x and dy at once (the parameter-gradient passes): each
// item widens and stores the block of both raw planes before its butterflies.
template <typename T>
__device__ __forceinline__ void widen_levels12_pair(const T* srca, float* sa, int spa, const WtBuf SA,
                                                    const WtBuf DA1, const WtBuf DA2, const T* srcb, float* sb,
                                                    int spb, const WtBuf SB, const WtBuf DB1, const WtBuf DB2,
                                                    int H, int W, float* dbase, int dps, int np, int H1, int W1,
                                                    int H2, int W2, const WtDiv& dpp, const WtDiv& dw, int tid,
                                                    int nthreads) {
  const int HW = H * W;
  const bool vec = (W & 3) == 0 && (SA.pcol & 3) == 0 && (SB.pcol & 3) == 0;
  const int per_plane = H2 * W2;
  for (int it = tid; it < np * per_plane; it += nthreads) {
    const int g = fdiv(it, dpp);
    const int rem = it - g * per_plane;
    const int P = fdiv(rem, dw);
    const int Q = rem - P * W2;
    float xa[4][4], xb[4][4];
    widen_block4<T>(srca + g * HW, H, W, P, Q, sa + g * spa, SA, vec, xa);
    widen_block4<T>(srcb + g * HW, H, W, P, Q, sb + g * spb, SB, vec, xb);
    float* ps = dbase + g * dps;
    store_block12(xa, ps, DA1, DA2, P, Q, H1, W1);
    store_block12(xb, ps, DB1, DB2, P, Q, H1, W1);
  }
}

// Widen np raw 16-bit planes (H*W elements each, consecutive in `src`, as the
// bulk copies leave them) into the float32 interiors of buffer B of each
// plane slot.  `per` elements per item: 4 when W % 4 == 0 (8-byte loads,
// 16-byte stores: B.pcol and B.stride are multiples of 4), 2 when W is even
// (4-byte loads, 8-byte stores), else 1; dpp and dw divide by the items per
// plane and per row.
template <typename T>
__device__ __forceinline__ void widen_planes(float* dbase, int dps, const WtBuf B, const T* src, int np, int H,
                                             int W, int per, const WtDiv& dpp, const WtDiv& dw, int tid,
                                             int nthreads) {
  const int HW = H * W;
  if (per == 2) {
    const int Wv = W >> 1;
    const int per_plane = H * Wv;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int j = (rem - i * Wv) << 1;
      const uint32_t raw = *reinterpret_cast<const uint32_t*>(src + g * HW + i * W + j);
      const T* h = reinterpret_cast<const T*>(&raw);
      *reinterpret_cast<float2*>(dbase + g * dps + B.off + (i + B.prow) * B.stride + j + B.pcol) =
          make_float2(to_f32(h[0]), to_f32(h[1]));
    }
  } else if (per == 4) {
    const int Wv = W >> 2;
    const int per_plane = H * Wv;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int j = (rem - i * Wv) << 2;
      const uint2 raw = *reinterpret_cast<const uint2*>(src + g * HW + i * W + j);
      const T* h = reinterpret_cast<const T*>(&raw);
      *reinterpret_cast<float4*>(dbase + g * dps + B.off + (i + B.prow) * B.stride + j + B.pcol) =
          make_float4(to_f32(h[0]), to_f32(h[1]), to_f32(h[2]), to_f32(h[3]));
    }
  } else {
    for (int it = tid; it < np * HW; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * HW;
      const int i = fdiv(rem, dw);
      const int j = rem - i * W;
      dbase[g * dps + B.off + (i + B.prow) * B.stride + j + B.pcol] = to_f32(src[it]);
    }
  }
}

// haar_levels12 for two same-sized pyramids at once (x and dy of the
// parameter-gradient pass): each item loads the block of both sources before
// any store, so the two butterfly chains overlap, and shares the indexing.
__device__ __forceinline__ void haar_levels12_pair(const float* sa, int spa, const WtBuf SA, const WtBuf DA1,
                                                   const WtBuf DA2, const float* sb, int spb, const WtBuf SB,
                                                   const WtBuf DB1, const WtBuf DB2, float* dbase, int dps,
                                                   int np, int H1, int W1, int H2, int W2, const WtDiv& dpp,
                                                   const WtDiv& dw, int tid, int nthreads) {
  const int per_plane = H2 * W2;
  for (int it = tid; it < np * per_plane; it += nthreads) {
    const int g = fdiv(it, dpp);
    const int rem = it - g * per_plane;
    const int P = fdiv(rem, dw);
    const int Q = rem - P * W2;
    float xa[4][4], xb[4][4];
    load_block4(sa + g * spa + SA.off + (4 * P + SA.prow) * SA.stride + 4 * Q + SA.pcol, SA, xa);
    load_block4(sb + g * spb + SB.off + (4 * P + SB.prow) * SB.stride + 4 * Q + SB.pcol, SB, xb);
    float* ps = dbase + g * dps;
    store_block12(xa, ps, DA1, DA2, P, Q, H1, W1);
    store_block12(xb, ps, DB1, DB2, P, Q, H1, W1);
  }
}

// haar_level for two same-sized pyramids at once (both sources read before
// any store).
__device__ __forceinline__ void haar_level_pair(const float* sbase, int sps, float* dbase, int dps, int np,
                                                const WtBuf SA, const WtBuf DA, const WtBuf SB, const WtBuf DB,
                                                int Hl, int Wl, const WtDiv& dpp, const WtDiv& dw, int tid,
                                                int nthreads) {
  const int per_plane = Hl * Wl;
  for (int it = tid; it < np * per_plane; it += nthreads) {
    const int g = fdiv(it, dpp);
    const int rem = it - g * per_plane;
    const int p = fdiv(rem, dw);
    const int q = rem - p * Wl;
    const float* s1 = sbase + g * sps + SA.off + (2 * p + SA.prow) * SA.stride + 2 * q + SA.pcol;
    const float* s2 = sbase + g * sps + SB.off + (2 * p + SB.prow) * SB.stride + 2 * q + SB.pcol;
    const float a1 = s1[0], b1 = s1[1], c1 = s1[SA.stride], d1 = s1[SA.stride + 1];
    const float a2 = s2[0], b2 = s2[1], c2 = s2[SB.stride], d2 = s2[SB.stride + 1];
    float o1[4], o2[4];
    butterfly4(a1, b1, c1, d1, o1);
    butterfly4(a2, b2, c2, d2, o2);
    float* t1 = dbase + g * dps + DA.off + (p + DA.prow) * DA.stride + q + DA.pcol;
    float* t2 = dbase + g * dps + DB.off + (p + DB.prow) * DB.stride + q + DB.pcol;
#pragma unroll
    for (int b = 0; b < 4; ++b) t1[b * DA.band] = o1[b];
#pragma unroll
    for (int b = 0; b < 4; ++b) t2[b * DB.band] = o2[b];
  }
}

// Copy planes n0 .. n0+np-1 of channel c from global memory into the
// interiors of buffer B of each plane slot.
template <typename T>
__device__ __forceinline__ void load_planes(float* dbase, int dps, const WtBuf B,
                                            const T* __restrict__ src, int n0, int np, int c, int C,
                                            int H, int W, bool vec, const WtDiv& dpp, const WtDiv& dw,
                                            int tid, int nthreads) {
  const size_t HW = (size_t)H * W;
  if (vec) {
    constexpr int V = Vec16<T>::N;
    const int Wv = W / V;
    const int per_plane = H * Wv;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int jv = rem - i * Wv;
      float v[V];
      ldg16<T>(src + ((size_t)(n0 + g) * C + c) * HW + (size_t)i * W + jv * V, v);
      float* d = dbase + g * dps + B.off + (i + B.prow) * B.stride + jv * V + B.pcol;
      if ((B.pcol & 3) == 0) {
#pragma unroll
        for (int e = 0; e < V; e += 4)
          *reinterpret_cast<float4*>(d + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
      } else {
#pragma unroll
        for (int e = 0; e < V; ++e) d[e] = v[e];
      }
    }
  } else {
    const int per_plane = H * W;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int j = rem - i * W;
      const float v = to_f32(src[((size_t)(n0 + g) * C + c) * HW + rem]);
      dbase[g * dps + B.off + (i + B.prow) * B.stride + j + B.pcol] = v;
    }
  }
}

// Zero-filled load of np windows: buffer element (i, j), i < Hv, j < Wv, of
// plane g is source element (oy + i, ox + j) of plane (n0 + g, c), or zero
// outside the H x W plane.  vec: 16-byte items (W and ox multiples of the item
// width, source 16-byte aligned), so an item lies wholly inside or wholly
// outside the plane; B.pcol and B.stride are multiples of 4.
template <typename T>
__device__ __forceinline__ void load_window(float* dbase, int dps, const WtBuf B, const T* __restrict__ src,
                                            int n0, int np, int c, int C, int H, int W, int oy, int ox, int Hv,
                                            int Wv, bool vec, const WtDiv& dpp, const WtDiv& dw, int tid,
                                            int nthreads) {
  const size_t HW = (size_t)H * W;
  if (vec) {
    constexpr int V = Vec16<T>::N;
    const int Wq = Wv / V;
    const int per_plane = Hv * Wq;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int jq = rem - i * Wq;
      const int gi = oy + i, gj = ox + jq * V;
      float v[V];
      if (gi >= 0 && gi < H && gj >= 0 && gj < W) {
        ldg16<T>(src + ((size_t)(n0 + g) * C + c) * HW + (size_t)gi * W + gj, v);
      } else {
#pragma unroll
        for (int e = 0; e < V; ++e) v[e] = 0.f;
      }
      float* d = dbase + g * dps + B.off + (i + B.prow) * B.stride + jq * V + B.pcol;
#pragma unroll
      for (int e = 0; e < V; e += 4) *reinterpret_cast<float4*>(d + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    }
  } else {
    const int per_plane = Hv * Wv;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int j = rem - i * Wv;
      const int gi = oy + i, gj = ox + j;
      const float v = (gi >= 0 && gi < H && gj >= 0 && gj < W)
                          ? to_f32(src[((size_t)(n0 + g) * C + c) * HW + (size_t)gi * W + gj])
                          : 0.f;
      dbase[g * dps + B.off + (i + B.prow) * B.stride + j + B.pcol] = v;
    }
  }
}

// Asynchronous copy of float32 planes n0 .. n0+np-1 of channel c into the
// interiors of buffer B (cp.async: global -> shared without registers).
// 16-byte copies when rows are 16-byte aligned in both spaces, else 4-byte.
// The caller commits and waits (cp_async_wait_all) before a barrier.
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

__device__ __forceinline__ void cp_async8(float* dst, const float* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d), "l"(src) : "memory");
}

// Copies with the widest granule G (4, 2 or 1 floats) that keeps both sides
// aligned: G = 4 needs 16-byte aligned rows in global memory (vec) and a
// buffer margin that is a multiple of 4 floats; G = 2 a margin that is even.
__device__ __forceinline__ void load_planes_async(float* dbase, int dps, const WtBuf B,
                                                  const float* __restrict__ src, int n0, int np, int c,
                                                  int C, int H, int W, bool vec, const WtDiv& dpp,
                                                  const WtDiv& dw, int tid, int nthreads) {
  const size_t HW = (size_t)H * W;
  if (vec) {  // W % 4 == 0 and 16-byte aligned rows: items are 4-float groups
    const int Wv = W >> 2;
    const int per_plane = H * Wv;
    const bool g4 = (B.pcol & 3) == 0, g2 = (B.pcol & 1) == 0;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int jv = rem - i * Wv;
      float* d = dbase + g * dps + B.off + (i + B.prow) * B.stride + 4 * jv + B.pcol;
      const float* sp = src + ((size_t)(n0 + g) * C + c) * HW + (size_t)i * W + 4 * jv;
      if (g4) {
        cp_async16(d, sp);
      } else if (g2) {
        cp_async8(d, sp);
        cp_async8(d + 2, sp + 2);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) cp_async4(d + e, sp + e);
      }
    }
  } else {
    const int per_plane = H * W;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = fdiv(it, dpp);
      const int rem = it - g * per_plane;
      const int i = fdiv(rem, dw);
      const int j = rem - i * W;
      cp_async4(dbase + g * dps + B.off + (i + B.prow) * B.stride + j + B.pcol,
                src + ((size_t)(n0 + g) * C + c) * HW + rem);
    }
  }
}

// ---- TMA plane loads (cp.async.bulk.tensor) with mbarrier completion ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// First 128-byte aligned float at or after p (shared memory); the launch
// reserves WT_SMEM_SLACK extra bytes for the shift.
__device__ __forceinline__ float* align_smem128(float* p) {
  return p + (((128u - (smem_u32(p) & 127u)) & 127u) >> 2);
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(mbar)), "r"(count) : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses (and
// mbarrier initialisation) before later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Makes this thread's mbarrier initialisations visible to the async proxy
// (and to the rest of the CTA after the next barrier).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(mbar)), "r"(bytes)
               : "memory");
}

// 4-D tiled tensor load: box at coordinates (c0, c1, c2, c3) into dst; the
// transfer signals complete_tx on mbar.  Out-of-range elements are zero.
__device__ __forceinline__ void tma_load_4d(float* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                           uint64_t* mbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(mbar))
      : "memory");
}

// Hint: bring the 4-D box at (c0, c1, c2, c3) of `map` into L2 (no shared
// memory, no completion to wait for; out-of-range parts are ignored).  A CTA
// with one input set issues it for the next unit as soon as the current
// unit's copy has landed, so the next copy, issued when the set is free
// again, is served from L2.
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];\n" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// Contiguous global -> shared bulk copy (both addresses 16-byte aligned, size
// a multiple of 16); completes `bytes` of transaction on mbar.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
               ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(mbar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* mbar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(mbar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of mbar to complete, giving up after about
// 2^shift clock cycles (shift = 31 in normal operation: about a second).
// Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* mbar, uint32_t parity, int shift) {
  const long long t0 = clock64();
  while (!mbar_try_wait(mbar, parity)) {
    if (clock64() - t0 > (1ll << shift)) return false;
  }
  return true;
}

__device__ __forceinline__ void zero_smem(float* sm, int nfloats, int tid, int nthreads) {
  float4* s4 = reinterpret_cast<float4*>(sm);
  for (int i = tid; i < (nfloats >> 2); i += nthreads) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace wt
