// Element-wise kernels of the coarse-level split (host logic in wtconv_api.cu).
//
// A layer whose tile window does not fit one CTA (large planes with a deep
// pyramid and a wide kernel) is computed as two layers.  Levels 1..s and the
// base convolution run on the full planes as usual.  Levels s+1..L depend on
// x only through its level-s low-pass band, and reach the output only
// through the level-s low-pass position of each pixel: in the collapsed
// synthesis a pixel (i, j) takes level l's coefficients at (i >> l, j >> l)
// with the sign bits (i >> (l-1)) & 1, (j >> (l-1)) & 1, and for l > s these
// are bits of (i >> s, j >> s).  So the coarse part of y is C[i >> s][j >> s],
// where C is the output of a WTConv2d layer with L - s levels (no base
// convolution) on the level-s low-pass planes.  These kernels build those
// planes (block sums: the unnormalised Haar low-pass of s levels) and add the
// coarse part back, replicated over each 2^s x 2^s block.  The transpose of
// the same chain gives the input gradient (block sums of dy, the rotated
// coarse layer, replication), and the coarse levels' parameter gradients
// are that layer's, on the low-pass planes of x and dy.
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805), technical summary, "Methodology": the
// synthesis collapsed into one sum indexed by the bits of the output
// coordinate ("Proposition 2"), which is what makes the coarse levels
// separable from the fine ones.  The split itself is this library's.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "wtconv_device.cuh"
#include "wtconv_launch.h"

namespace wt {

namespace {

constexpr int kSplitThreads = 256;
constexpr int kChunk = 4096;  // columns per shared-memory pass (a multiple of every block width 2^s, s <= 7)

// ll[r][Q] = sum of the 2^s x 2^s block of x at (P 2^s, Q 2^s), r = plane * Hs + P;
// pixels past the plane count as zero.  One CTA per low-pass row: the
// threads sum columns over the block's rows (coalesced), then blocks of
// columns in shared memory.
template <typename T>
__global__ void __launch_bounds__(kSplitThreads)
    lowpass_kernel(const T* __restrict__ x, float* __restrict__ ll, long long rows, int H, int W, int s, int Hs,
                   int Ws) {
  __shared__ float colsum[kChunk];
  const int B = 1 << s;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const long long plane = r / Hs;
    const int P = (int)(r - plane * Hs);
    const T* src = x + plane * (long long)H * W;
    const int i0 = P << s, i1 = min(i0 + B, H);
    for (int c0 = 0; c0 < W; c0 += kChunk) {
      const int c1 = min(c0 + kChunk, W);
      for (int j = c0 + threadIdx.x; j < c1; j += blockDim.x) {
        float v = 0.f;
        for (int i = i0; i < i1; ++i) v += to_f32(src[(long long)i * W + j]);
        colsum[j - c0] = v;
      }
      __syncthreads();
      const int q1 = (c1 + B - 1) >> s;
      for (int Q = (c0 >> s) + threadIdx.x; Q < q1; Q += blockDim.x) {
        const int j0 = Q << s, j1 = min(j0 + B, W);
        float v = 0.f;
        for (int j = j0; j < j1; ++j) v += colsum[j - c0];
        ll[r * Ws + Q] = v;
      }
      __syncthreads();
    }
  }
}

// y[plane][i][j] += c[plane][i >> s][j >> s], in float32, rounded to T once.
template <typename T>
__global__ void __launch_bounds__(kSplitThreads)
    add_carry_kernel(T* __restrict__ y, const float* __restrict__ c, long long rows, int H, int W, int s, int Hs,
                     int Ws) {
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {  // r = plane * H + i
    const long long plane = r / H;
    const int i = (int)(r - plane * H);
    T* dst = y + r * W;
    const float* src = c + (plane * Hs + (i >> s)) * Ws;
    for (int j = threadIdx.x; j < W; j += blockDim.x) dst[j] = from_f32<T>(to_f32(dst[j]) + src[j >> s]);
  }
}

__global__ void scale_kernel(const float* __restrict__ in, float* __restrict__ out, int n, float f) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) out[i] = in[i] * f;
}

unsigned grid_for(long long rows) {
  const long long cap = 8LL * (sm_count() > 0 ? sm_count() : 152);
  return (unsigned)(rows < cap ? (rows > 0 ? rows : 1) : cap);
}

}  // namespace

cudaError_t launch_lowpass(int dtype, const void* x, float* ll, long long planes, int H, int W, int s,
                           cudaStream_t stream) {
  const int Hs = (int)(((long long)H + (1LL << s) - 1) >> s), Ws = (int)(((long long)W + (1LL << s) - 1) >> s);
  const long long rows = planes * Hs;
  if (rows == 0) return cudaSuccess;
  const unsigned g = grid_for(rows);
  if (dtype == 0)
    lowpass_kernel<float><<<g, kSplitThreads, 0, stream>>>(static_cast<const float*>(x), ll, rows, H, W, s, Hs, Ws);
  else if (dtype == 1)
    lowpass_kernel<__half><<<g, kSplitThreads, 0, stream>>>(static_cast<const __half*>(x), ll, rows, H, W, s, Hs, Ws);
  else
    lowpass_kernel<__nv_bfloat16><<<g, kSplitThreads, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), ll, rows, H,
                                                                    W, s, Hs, Ws);
  return cudaGetLastError();
}

cudaError_t launch_add_carry(int dtype, void* y, const float* c, long long planes, int H, int W, int s,
                             cudaStream_t stream) {
  const int Hs = (int)(((long long)H + (1LL << s) - 1) >> s), Ws = (int)(((long long)W + (1LL << s) - 1) >> s);
  const long long rows = planes * H;
  if (rows == 0) return cudaSuccess;
  const unsigned g = grid_for(rows);
  if (dtype == 0)
    add_carry_kernel<float><<<g, kSplitThreads, 0, stream>>>(static_cast<float*>(y), c, rows, H, W, s, Hs, Ws);
  else if (dtype == 1)
    add_carry_kernel<__half><<<g, kSplitThreads, 0, stream>>>(static_cast<__half*>(y), c, rows, H, W, s, Hs, Ws);
  else
    add_carry_kernel<__nv_bfloat16><<<g, kSplitThreads, 0, stream>>>(static_cast<__nv_bfloat16*>(y), c, rows, H, W,
                                                                     s, Hs, Ws);
  return cudaGetLastError();
}

cudaError_t launch_scale(const float* in, float* out, int n, float f, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int blocks = (n + kSplitThreads - 1) / kSplitThreads;
  scale_kernel<<<blocks < 1024 ? blocks : 1024, kSplitThreads, 0, stream>>>(in, out, n, f);
  return cudaGetLastError();
}

}  // namespace wt
