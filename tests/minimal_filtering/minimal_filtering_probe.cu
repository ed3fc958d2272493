// Minimal filtering against the direct form, for the k x k depthwise
// convolution tiles of the WTConv2d layer (k = 5): a measurement, not part of
// the library (test infrastructure).
//
// The layer's band and base convolutions are depthwise: every channel has
// its own 5 x 5 kernel and one input plane, so a transformed input tile
// serves one kernel only.  Minimal filtering (Lavin & Gray, "Fast Algorithms
// for Convolutional Neural Networks", CVPR 2016) trades multiplies for
// transform additions, which run on the same FP32 pipe.  This program times,
// on the same shared-memory planes and thread tiles, three forms of one
// thread computing TH = 4, 8 or 16 output rows x 4 output columns of a 64 x 64 plane
// (same padding):
//   direct   25 FMAs per output, the form the library's kernels use;
//   F(2, 5)  along rows: two 6-point input transforms per input row,
//            5 x 6 products per output row and segment, one 2-output
//            transform per segment;
//   F(4, 5)  along rows: one 8-point input transform per input row,
//            5 x 8 products per output row, one 4-output transform.
// The transforms come from winograd_transforms.h (gen_transforms.py); the
// symmetric row pairs of B^T and column pairs of A^T are applied in their
// even/odd factored form (two partial sums, then their sum and difference).
//
// Usage:  minimal_filtering_probe            numerics (rel-L2 against a double
//                                            direct sum) and timings
//         minimal_filtering_probe check      numerics only
// Exit status 0 when every form's rel-L2 is within its bound.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <vector>

#include "winograd_transforms.h"

#define CK(x)                                                                                  \
  do {                                                                                         \
    cudaError_t e_ = (x);                                                                      \
    if (e_ != cudaSuccess) {                                                                   \
      printf("CUDA error %s at %s:%d\n", cudaGetErrorString(e_), __FILE__, __LINE__);          \
      return 2;                                                                                \
    }                                                                                          \
  } while (0)

constexpr int kP = 64;           // plane side
constexpr int kS = kP + 4;       // shared row stride (2 zero columns on each side)
constexpr int kWStride = 40;     // floats of per-channel weights (the largest form: 5 x 8)

// The n-point input transform v = BT d.  Row 0 and row n-1 are summed
// directly; rows (1, 2), (3, 4), ... are pairs whose odd-column entries
// differ in sign, formed as (even part) +- (odd part).
template <int N>
__device__ __forceinline__ float bt(int i, int j) { return N == 8 ? kBT4(i, j) : kBT2(i, j); }
template <int M>
__device__ __forceinline__ float at(int i, int j) { return M == 4 ? kAT4(i, j) : kAT2(i, j); }

template <int N>
__device__ __forceinline__ void input_transform(const float* d, float* v) {
#pragma unroll
  for (int t = 0; t < N; t += (t == 0 || t == N - 1) ? 1 : 2) {
    if (t == 0 || t == N - 1) {
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < N; ++j)
        if (bt<N>(t, j) != 0.f) s = fmaf(bt<N>(t, j), d[j], s);
      v[t] = s;
    } else {
      float e = 0.f, o = 0.f;
#pragma unroll
      for (int j = 0; j < N; ++j)
        if (bt<N>(t, j) != 0.f) {
          if (j % 2 == 0) e = fmaf(bt<N>(t, j), d[j], e);
          else o = fmaf(bt<N>(t, j), d[j], o);
        }
      v[t] = e + o;
      v[t + 1] = e - o;
    }
  }
}

// y = AT m for M outputs from N products: column pairs (1, 2), (3, 4), ...
// enter as their sum (even outputs) or difference (odd outputs).
template <int M, int N>
__device__ __forceinline__ void output_transform(const float* m, float* y) {
  float p[N], q[N];
#pragma unroll
  for (int t = 1; t + 1 < N; t += 2) {
    p[t] = m[t] + m[t + 1];
    q[t] = m[t] - m[t + 1];
  }
#pragma unroll
  for (int i = 0; i < M; ++i) {
    float s = 0.f;
    if (at<M>(i, 0) != 0.f) s = fmaf(at<M>(i, 0), m[0], s);
#pragma unroll
    for (int t = 1; t + 1 < N; t += 2)
      if (at<M>(i, t) != 0.f) s = fmaf(at<M>(i, t), i % 2 == 0 ? p[t] : q[t], s);
    if (at<M>(i, N - 1) != 0.f) s = fmaf(at<M>(i, N - 1), m[N - 1], s);
    y[i] = s;
  }
}

// FORM 0 direct, 2 = F(2, 5), 4 = F(4, 5).  Block: 16 x (64 / TH) threads,
// one tile each; block b convolves plane b with `chans` kernels.
template <int FORM, int TH, bool STORE>
__global__ void __launch_bounds__(16 * (kP / TH)) tile_kernel(const float* __restrict__ planes,
                                                              const float* __restrict__ wts, int chans,
                                                              float* __restrict__ out) {
  __shared__ __align__(16) float s[kS * kS];
  const float* src = planes + (size_t)blockIdx.x * kP * kP;
  for (int i = threadIdx.x; i < kS * kS; i += blockDim.x) {
    const int r = i / kS - 2, c = i % kS - 2;
    s[i] = (r >= 0 && r < kP && c >= 0 && c < kP) ? src[r * kP + c] : 0.f;
  }
  __syncthreads();
  const int r0 = (threadIdx.x / 16) * TH, c0 = (threadIdx.x % 16) * 4;
  constexpr int NV = FORM == 0 ? 8 : FORM == 2 ? 6 : 8;  // transformed points per segment
  constexpr int NSEG = FORM == 2 ? 2 : 1;
  constexpr int NACC = FORM == 0 ? 4 : NSEG * NV;
  float chk = 0.f;
  for (int ch = 0; ch < chans; ++ch) {
    float w[FORM == 0 ? 25 : 5 * NV];
    const float* wc = wts + (size_t)ch * kWStride;
#pragma unroll
    for (int i = 0; i < (FORM == 0 ? 25 : 5 * NV); ++i) w[i] = __ldg(wc + i);
    float acc[TH][NACC];
#pragma unroll
    for (int o = 0; o < TH; ++o)
#pragma unroll
      for (int a = 0; a < NACC; ++a) acc[o][a] = 0.f;
#pragma unroll
    for (int r = 0; r < TH + 4; ++r) {
      float d[8];
      const float4 lo = *reinterpret_cast<const float4*>(&s[(r0 + r) * kS + c0]);
      const float4 hi = *reinterpret_cast<const float4*>(&s[(r0 + r) * kS + c0 + 4]);
      d[0] = lo.x; d[1] = lo.y; d[2] = lo.z; d[3] = lo.w;
      d[4] = hi.x; d[5] = hi.y; d[6] = hi.z; d[7] = hi.w;
      if constexpr (FORM == 0) {
#pragma unroll
        for (int o = 0; o < TH; ++o) {
          const int kr = r - o;
          if (kr < 0 || kr > 4) continue;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int kc = 0; kc < 5; ++kc) acc[o][c] = fmaf(w[kr * 5 + kc], d[c + kc], acc[o][c]);
        }
      } else {
        float v[NSEG * NV];
        if constexpr (FORM == 4) {
          input_transform<8>(d, v);
        } else {
          input_transform<6>(d, v);
          input_transform<6>(d + 2, v + 6);
        }
#pragma unroll
        for (int o = 0; o < TH; ++o) {
          const int kr = r - o;
          if (kr < 0 || kr > 4) continue;
#pragma unroll
          for (int a = 0; a < NSEG * NV; ++a) acc[o][a] = fmaf(w[kr * NV + a % NV], v[a], acc[o][a]);
        }
      }
    }
#pragma unroll
    for (int o = 0; o < TH; ++o) {
      float y[4];
      if constexpr (FORM == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) y[c] = acc[o][c];
      } else if constexpr (FORM == 4) {
        output_transform<4, 8>(acc[o], y);
      } else {
        output_transform<2, 6>(acc[o], y);
        output_transform<2, 6>(acc[o] + 6, y + 2);
      }
      if constexpr (STORE) {
        float* dst = out + (((size_t)blockIdx.x * chans + ch) * kP + r0 + o) * kP + c0;
        *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
      } else {
        chk += (y[0] + y[1]) + (y[2] + y[3]);
      }
    }
  }
  if constexpr (!STORE) out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = chk;
}

template <int FORM, int TH, bool STORE>
static cudaError_t launch(int blocks, const float* planes, const float* wts, int chans, float* out) {
  tile_kernel<FORM, TH, STORE><<<blocks, 16 * (kP / TH)>>>(planes, wts, chans, out);
  return cudaGetLastError();
}

static uint64_t g_rng = 0x9E3779B97F4A7C15ull;
static double uniform() {  // splitmix64 -> [0, 1)
  uint64_t z = (g_rng += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (double)(z >> 11) * (1.0 / 9007199254740992.0);
}
static double normal() {  // Box-Muller
  double u1 = uniform(), u2 = uniform();
  if (u1 < 1e-300) u1 = 1e-300;
  return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
}

// Per-channel weights in each form's layout: g (5 x 5), or U = G g along
// rows (5 x NV), computed in double and rounded once.
static void weights(int form, const std::vector<double>& g, int chans, std::vector<float>& w) {
  w.assign((size_t)chans * kWStride, 0.f);
  for (int ch = 0; ch < chans; ++ch) {
    const double* gc = &g[(size_t)ch * 25];
    float* wc = &w[(size_t)ch * kWStride];
    if (form == 0) {
      for (int i = 0; i < 25; ++i) wc[i] = (float)gc[i];
    } else {
      const int nv = form == 2 ? 6 : 8;
      for (int kr = 0; kr < 5; ++kr)
        for (int t = 0; t < nv; ++t) {
          double u = 0;
          for (int k = 0; k < 5; ++k) u += (double)(form == 2 ? kG2(t, k) : kG4(t, k)) * gc[kr * 5 + k];
          wc[kr * nv + t] = (float)u;
        }
    }
  }
}

template <int FORM, int TH>
static int run_form(const char* name, bool time_it, const float* d_planes, const std::vector<float>& h_planes,
                    const std::vector<double>& g, int vblocks, int vchans, int tblocks, int tchans, double bound,
                    bool* ok) {
  std::vector<float> w;
  weights(FORM, g, std::max(vchans, tchans), w);
  float *d_w = nullptr, *d_out = nullptr;
  const size_t vout = (size_t)vblocks * vchans * kP * kP;
  const size_t tout = (size_t)tblocks * 16 * (kP / TH);
  CK(cudaMalloc(&d_w, w.size() * sizeof(float)));
  CK(cudaMalloc(&d_out, std::max(vout, tout) * sizeof(float)));
  CK(cudaMemcpy(d_w, w.data(), w.size() * sizeof(float), cudaMemcpyHostToDevice));
  // Numerics: every output of vblocks planes x vchans kernels against a double direct sum.
  CK((launch<FORM, TH, true>(vblocks, d_planes, d_w, vchans, d_out)));
  CK(cudaDeviceSynchronize());
  std::vector<float> y(vout);
  CK(cudaMemcpy(y.data(), d_out, vout * sizeof(float), cudaMemcpyDeviceToHost));
  double num = 0, den = 0;
  for (int b = 0; b < vblocks; ++b)
    for (int ch = 0; ch < vchans; ++ch)
      for (int i = 0; i < kP; ++i)
        for (int j = 0; j < kP; ++j) {
          double ref = 0;
          for (int a = 0; a < 5; ++a)
            for (int c = 0; c < 5; ++c) {
              const int ii = i + a - 2, jj = j + c - 2;
              if (ii < 0 || ii >= kP || jj < 0 || jj >= kP) continue;
              ref += g[(size_t)ch * 25 + a * 5 + c] * (double)h_planes[((size_t)b * kP + ii) * kP + jj];
            }
          const double e = y[(((size_t)b * vchans + ch) * kP + i) * kP + j] - ref;
          num += e * e;
          den += ref * ref;
        }
  const double rel = std::sqrt(num / den);
  const bool pass = rel <= bound;
  *ok = *ok && pass;
  printf("%-8s TH=%d  rel-L2 %.3e (bound %.0e) %s", name, TH, rel, bound, pass ? "ok" : "FAIL");
  if (time_it) {
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    for (int i = 0; i < 3; ++i) CK((launch<FORM, TH, false>(tblocks, d_planes, d_w, tchans, d_out)));
    std::vector<float> ms;
    for (int rep = 0; rep < 7; ++rep) {
      CK(cudaEventRecord(e0));
      CK((launch<FORM, TH, false>(tblocks, d_planes, d_w, tchans, d_out)));
      CK(cudaEventRecord(e1));
      CK(cudaEventSynchronize(e1));
      float t = 0;
      CK(cudaEventElapsedTime(&t, e0, e1));
      ms.push_back(t);
    }
    std::sort(ms.begin(), ms.end());
    const double t = ms[ms.size() / 2] * 1e-3;
    const double outputs = (double)tblocks * tchans * kP * kP;
    cudaFuncAttributes fa;
    CK(cudaFuncGetAttributes(&fa, tile_kernel<FORM, TH, false>));
    int dev = 0, sms = 0, clk_khz = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CK(cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, dev));
    const double peak_fma = (double)sms * 128 * clk_khz * 1e3;  // FP32 FMA/s at the reported clock
    printf("  |  %.3f ms  %.2f Goutput/s  direct-equivalent FMA rate %.1f %% of FP32 peak  (%d regs)",
           t * 1e3, outputs / t * 1e-9, 100.0 * outputs * 25 / t / peak_fma, fa.numRegs);
    CK(cudaEventDestroy(e0));
    CK(cudaEventDestroy(e1));
  }
  printf("\n");
  CK(cudaFree(d_w));
  CK(cudaFree(d_out));
  return 0;
}

int main(int argc, char** argv) {
  const bool time_it = !(argc > 1 && strcmp(argv[1], "check") == 0);
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int vblocks = 6, vchans = 4;
  const int tblocks = sms * 8, tchans = 64;  // timed: planes L2-resident, 64 kernels per plane
  const int nplanes = std::max(vblocks, tblocks);
  std::vector<float> planes((size_t)nplanes * kP * kP);
  for (auto& v : planes) v = (float)normal();
  std::vector<double> g((size_t)std::max(vchans, tchans) * 25);
  for (auto& v : g) v = (double)(float)(0.05 * normal());  // float-representable, as the direct form uses them
  float* d_planes = nullptr;
  CK(cudaMalloc(&d_planes, planes.size() * sizeof(float)));
  CK(cudaMemcpy(d_planes, planes.data(), planes.size() * sizeof(float), cudaMemcpyHostToDevice));
  printf("5 x 5 depthwise tiles of 64 x 64 planes: %d planes x %d kernels timed, %d SMs\n", tblocks, tchans, sms);
  bool ok = true;
  // Bounds: the direct form is a float32 sum of 25 products; the transforms
  // add their own rounding (F(4, 5) more: 8-point transforms with entries up
  // to 5.25 and down to 1/360).
  if (run_form<0, 4>("direct", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-6, &ok)) return 2;
  if (run_form<0, 8>("direct", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-6, &ok)) return 2;
  if (run_form<0, 16>("direct", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-6, &ok)) return 2;
  if (run_form<2, 4>("F(2,5)", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-5, &ok)) return 2;
  if (run_form<2, 8>("F(2,5)", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-5, &ok)) return 2;
  if (run_form<4, 4>("F(4,5)", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-4, &ok)) return 2;
  if (run_form<4, 8>("F(4,5)", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-4, &ok)) return 2;
  if (run_form<4, 16>("F(4,5)", time_it, d_planes, planes, g, vblocks, vchans, tblocks, tchans, 1e-4, &ok)) return 2;
  CK(cudaFree(d_planes));
  printf("%s\n", ok ? "all forms within bounds" : "a form exceeded its bound");
  return ok ? 0 : 1;
}
