// Device building blocks of libwtconv (sm_103a).
//
// Depthwise convolution and Haar butterflies are not dense contractions, so
// everything here runs on the FP32 pipes: tiles of outputs per thread with
// register-resident weights and sliding rows read from shared memory with
// 16-byte loads.
#pragma once

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

// acc[du*K+dv] += sum_{o,j} d[o][j] * win[(o+du)*stride + j+dv]   (weight-gradient correlation)
// Returns the sum of the d tile (for the bias gradient).
template <int K, int TR, int TC>
__device__ __forceinline__ float corr_tile(const float* __restrict__ win, int wstride,
                                           const float* __restrict__ dsrc, int dstride,
                                           float (&acc)[K * K]) {
  constexpr int NV = (TC + K - 1 + 3) / 4;
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
    float seg[4 * NV];
    lds_row<NV>(win + a * wstride, seg);
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

// One Haar analysis level on the planes g < np of a CTA:
//   dst_b[p][q] = sum_{u,v} sign_b(u,v) * src[2p+u][2q+v],  p < Hl, q < Wl
// (unnormalised: the 1/2 per level is folded into the weights).  Reads past
// the source interior hit its zero margin.
__device__ __forceinline__ void haar_level(float* sm, int plane_floats, int np, const WtBuf S,
                                           const WtBuf D, int Hl, int Wl, int tid, int nthreads) {
  const int per_plane = Hl * Wl;
  for (int it = tid; it < np * per_plane; it += nthreads) {
    const int g = it / per_plane;
    const int rem = it - g * per_plane;
    const int p = rem / Wl;
    const int q = rem - p * Wl;
    const float* s = sm + g * plane_floats + S.off + (2 * p + S.pad) * S.stride + 2 * q + S.pad;
    const float a = s[0], b = s[1], c = s[S.stride], d = s[S.stride + 1];
    const float s0 = a + b, d0 = a - b, s1 = c + d, d1 = c - d;
    float* o = sm + g * plane_floats + D.off + (p + D.pad) * D.stride + q + D.pad;
    o[0] = s0 + s1;           // low-pass
    o[D.band] = s0 - s1;      // row-high:    sign (-1)^u
    o[2 * D.band] = d0 + d1;  // column-high: sign (-1)^v
    o[3 * D.band] = d0 - d1;  // diagonal:    sign (-1)^(u+v)
  }
}

// Copy planes n0 .. n0+np-1 of channel c from global memory into the
// interiors of buffer B of each plane slot.
template <typename T>
__device__ __forceinline__ void load_planes(float* sm, int plane_floats, const WtBuf B,
                                            const T* __restrict__ src, int n0, int np, int c, int C,
                                            int H, int W, bool vec, int tid, int nthreads) {
  const size_t HW = (size_t)H * W;
  if (vec) {
    constexpr int V = Vec16<T>::N;
    const int Wv = W / V;
    const int per_plane = H * Wv;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = it / per_plane;
      const int rem = it - g * per_plane;
      const int i = rem / Wv;
      const int jv = rem - i * Wv;
      float v[V];
      ldg16<T>(src + ((size_t)(n0 + g) * C + c) * HW + (size_t)i * W + jv * V, v);
      float* d = sm + g * plane_floats + B.off + (i + B.pad) * B.stride + jv * V + B.pad;
#pragma unroll
      for (int e = 0; e < V; ++e) d[e] = v[e];
    }
  } else {
    const int per_plane = H * W;
    for (int it = tid; it < np * per_plane; it += nthreads) {
      const int g = it / per_plane;
      const int rem = it - g * per_plane;
      const int i = rem / W;
      const int j = rem - i * W;
      const float v = to_f32(src[((size_t)(n0 + g) * C + c) * HW + rem]);
      sm[g * plane_floats + B.off + (i + B.pad) * B.stride + j + B.pad] = v;
    }
  }
}

__device__ __forceinline__ void zero_smem(float* sm, int nfloats, int tid, int nthreads) {
  float4* s4 = reinterpret_cast<float4*>(sm);
  for (int i = tid; i < (nfloats >> 2); i += nthreads) s4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

}  // namespace wt
