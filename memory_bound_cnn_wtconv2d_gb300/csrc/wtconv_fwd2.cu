// Pipelined whole-plane WTConv2d forward pass and input-gradient pass
// (sm_103a).
//
// Paper: "Fast and Memory-Efficient Wavelet Convolutions via I/O-Aware
// Reformulation" (arXiv 2608.10805), technical summary, "Methodology": the
// Haar analysis is recomputed on chip, the per-channel scales are folded
// into the weights (and the base scale into the bias), and the multi-level
// synthesis collapses into one sum over levels indexed by the output
// coordinate's bits.  Here the sum is split in two: the levels 2..L are
// folded, on chip, into one level-1 term R1 by the synthesis cascade of the
// small coarse bands (pure adds, the 2^-l factors are folded into the
// weights), and the final strips add the level-1 butterfly of Z1 + R1 per
// output pixel.  Every activation crosses HBM once: x is read, y written.
//
// Work split inside a CTA (see wtconv_f2.h): a producer warp group prepares
// unit v+1 (plane copies, analysis, coarse levels) while the consumer warp
// group computes unit v (level-1 band convolutions, then the final strips:
// base convolution + synthesis + store).  The consumers' work is the bulk of
// the FMAs; they never wait on the analysis latency, and their strips are
// 4 x F2_SA register tiles read through 16-byte windows with conflict-free
// strides.
//
// The input-gradient pass is the same kernel with every kernel rotated by
// 180 degrees and no bias (A^T of the layer map; the Haar pair is
// orthonormal and k is odd).
#include "wtconv_f2.h"
#include "wtconv_fwd_tiles.cuh"
#include "wtconv_launch.h"

namespace wt {

// Bounded waits that gave up; read by take_fwd2_faults().
static __device__ unsigned int g_fwd2_faults;

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// Arrives at named barrier `id` (of n threads) without waiting: the
// signalling side of a producer/consumer handoff; the waiting side calls
// named_bar (bar.sync), which sleeps in hardware until all n have arrived.
__device__ __forceinline__ void named_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}

// Named barriers: 1 producer group, 2 consumer group; the handoffs between
// the groups (all F2_NT threads): producer -> consumer "X, B1 and the weights
// of unit v are ready" and "R1 of unit v is ready"; consumer -> producer "B1
// of unit v has been read".
#define F2_BAR_B1READY 3
#define F2_BAR_FREADY 4
#define F2_BAR_MID 5

// One try_wait that may suspend the thread until the phase completes or
// about `hint_ns` nanoseconds pass; a suspended warp issues nothing, so the
// warps that are still working keep the issue slots.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* mbar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(mbar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Waits for the phase of parity `parity` of mbar to complete, for at most
// 2^shift clock cycles.  Returns false if it gave up.
__device__ __forceinline__ bool f2_wait(uint64_t* mbar, uint32_t parity, int shift) {
  const long long t0 = clock64();
  while (!mbar_try_wait_hint(mbar, parity, 100000u)) {
    if (clock64() - t0 > (1ll << shift)) return false;
  }
  return true;
}

__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

// acc[o][j] += sum_{du,dv} w[du][dv] * win[(o + du) * S + j + dv] for a strip
// of SA x 4 outputs; `win` is 16-byte aligned, rows are read as NV float4s.
template <int K, int SA = F2_SA>
__device__ __forceinline__ void f2_strip(const float* __restrict__ win, int S, const float (&w)[K * K],
                                         float (&acc)[SA][4]) {
  constexpr int NV = (K + 6) / 4;
#pragma unroll
  for (int a = 0; a < SA + K - 1; ++a) {
    float seg[4 * NV];
    lds_row<NV>(win + a * S, seg);
#pragma unroll
    for (int o = 0; o < SA; ++o) {
      const int du = a - o;
      if (du >= 0 && du < K) {
#pragma unroll
        for (int dv = 0; dv < K; ++dv)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[o][j] = fmaf(w[du * K + dv], seg[j + dv], acc[o][j]);
      }
    }
  }
}

template <int K>
__device__ __forceinline__ void f2_load_w(const float* __restrict__ src, float (&w)[K * K]) {
  load_weights<K>(src, w);
}

// Element (i, j) of raw plane `rp` (H x W, type T, dense), 0 outside.
template <typename T>
__device__ __forceinline__ float raw_at(const T* rp, int i, int j, int H, int W) {
  return (i < H && j < W) ? to_f32(rp[i * W + j]) : 0.f;
}

// Four consecutive raw elements of row i from column j (j % 4 == 0, j + 3 < W,
// W % 4 == 0: the row segment is 16-byte (float) or 8-byte (16-bit) aligned).
template <typename T>
__device__ __forceinline__ void raw_vec4(const T* rp, int i, int j, int W, float (&v)[4]) {
  if constexpr (sizeof(T) == 4) {
    const float4 t = *reinterpret_cast<const float4*>(rp + i * W + j);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(rp + i * W + j);
    const T* h = reinterpret_cast<const T*>(&u);
    v[0] = to_f32(h[0]); v[1] = to_f32(h[1]); v[2] = to_f32(h[2]); v[3] = to_f32(h[3]);
  }
}

template <int K, typename T, bool ROT>
__global__ void __launch_bounds__(F2_NT, 2)
    fwd2_kernel(const __grid_constant__ WtF2Plan pl, const T* __restrict__ x, const float* __restrict__ w_base,
                const float* __restrict__ b_base, const float* __restrict__ w_sub, const float* __restrict__ s_base,
                const float* __restrict__ s_w, T* __restrict__ y) {
  extern __shared__ __align__(16) float sm_raw[];
  float* const sm = align_smem128(sm_raw);
  constexpr int R = K / 2;
  constexpr int KK = K * K;
  constexpr int SH = (4 - R) & 3;       // final strips' left shift (f2_sh)
  constexpr int ZO = SH == 2 ? 1 : 0;   // Z1 / R1 column offset (f2_zo)
  const int tid = threadIdx.x;
  const int C = pl.C, L = pl.L, P = pl.P, H = pl.H, W = pl.W;
  const int u0 = (int)((long long)pl.units * blockIdx.x / gridDim.x);
  const int u1 = (int)((long long)pl.units * (blockIdx.x + 1) / gridDim.x);
  const int nu = u1 - u0;
  uint64_t* const mb = reinterpret_cast<uint64_t*>(sm + pl.mb_off);
  uint64_t* const rawfull = mb;      // [2]: raw slot landed (bulk copies)
  __shared__ int s_abort;            // a copy did not land in time: the rest of the work is skipped

  // Every margin of every buffer is zero and stays zero: later writes touch
  // interiors only.  (The raw slots, written by the copies, need no zeros.)
  zero_smem(sm + pl.X.off, pl.mb_off - pl.X.off, tid, F2_NT);
  if (tid == 0) {
    mbar_init(&rawfull[0], 1);
    mbar_init(&rawfull[1], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  if (nu <= 0) return;

  if (tid < F2_NF) {
    // ======================= producer group =======================
    const int ft = tid;
    const bool bulk = pl.load_mode == 0;
    // Copies of unit v's raw planes into raw slot v & 1.
    auto issue = [&](int v) {
      const int u = u0 + v;
      const int c = wt_fdiv(u, pl.d_G);
      const int n0 = (u - c * pl.G) * P;
      const int np = min(P, pl.N - n0);
      char* dst = reinterpret_cast<char*>(sm + pl.raw_off + (v & 1) * pl.raw_slot);
      const char* src = reinterpret_cast<const char*>(x);
      const size_t pstride = (size_t)C * pl.plane_bytes;  // bytes between planes n and n+1 of a channel
      const size_t base = ((size_t)n0 * C + c) * pl.plane_bytes;
      if (bulk) {
        if (ft == 0) {
          fence_proxy_async();  // earlier generic reads of the slot precede the copies
          mbar_arrive_expect_tx(&rawfull[v & 1], (uint32_t)np * pl.plane_bytes + pl.dbg_extra_tx);
          for (int g = 0; g < np; ++g)
            bulk_load(dst + g * pl.raw_pb, src + base + g * pstride, (uint32_t)pl.plane_bytes, &rawfull[v & 1]);
        }
      } else {
        const int per = pl.plane_bytes / pl.chunk;
        for (int i = ft; i < np * per; i += F2_NF) {
          const int g = wt_fdiv(i, pl.d_chunks);
          const int o = (i - g * per) * pl.chunk;
          float* d = reinterpret_cast<float*>(dst + g * pl.raw_pb + o);
          const float* s = reinterpret_cast<const float*>(src + base + g * pstride + o);
          if (pl.chunk == 16) cp_async16(d, s);
          else if (pl.chunk == 8) cp_async8(d, s);
          else cp_async4(d, s);
        }
        cp_async_commit();
      }
    };
    // Copies issued and waited for, per raw slot (a slot has at most one copy
    // in flight): after a failed wait the remaining copies are still waited
    // for before the CTA exits.
    int issued0 = 0, issued1 = 0, waited0 = 0, waited1 = 0;
    auto issue_count = [&](int v) {
      issue(v);
      if (v & 1) ++issued1;
      else ++issued0;
    };
    issue_count(0);
    if (nu > 1) issue_count(1);
    int wch0 = -1, wch1 = -1;  // channel whose folded weights sit in slot 0 / 1
    bool dead = false;         // uniform over the group: the work of the remaining units is skipped
    for (int v = 0; v < nu; ++v) {
      const int u = u0 + v;
      const int c = wt_fdiv(u, pl.d_G);
      const int n0 = (u - c * pl.G) * P;
      const int np = min(P, pl.N - n0);
      const int slot = v & 1;
      bool ok = true;
      if (!dead) {
        if (bulk) {
          ok = f2_wait(&rawfull[slot], (uint32_t)(v >> 1) & 1u, pl.wait_shift);
          if (slot) ++waited1;
          else ++waited0;
        } else {
          if (v + 1 < nu) cp_async_wait_1();  // unit v+1's group may still be in flight
          else cp_async_wait_all();
        }
      }
      if (v >= 1) named_bar(F2_BAR_MID, F2_NT);  // the consumers have read B1 of unit v-1
      if (!ok) s_abort = 1;
      named_bar(1, F2_NF);
      if (!dead && s_abort) {
        dead = true;
        if (ft == 0) atomicAdd(&g_fwd2_faults, 1u);
      }
      float* const wsl = sm + pl.w_off + slot * pl.wslot;
      if (!dead && (slot ? wch1 : wch0) != c) {
        stage_weights<K, ROT>(wsl, pl.wb, L, C, c, w_base, w_sub, s_base, s_w, ft, F2_NF);
        if (slot) wch1 = c;
        else wch0 = c;
      }
      // (1) analysis of 4x4 input blocks: the float32 plane X, the level-1
      // bands B1 and (L >= 2) the level-2 bands B2.
      {
        const T* rawb = reinterpret_cast<const T*>(reinterpret_cast<const char*>(sm + pl.raw_off + slot * pl.raw_slot));
        const bool vec = (W & 3) == 0;
        const WtF2Buf XB = pl.X, B1 = pl.B[1], B2 = pl.B[2];
        const int xo = pl.X.off + slot * pl.xslot;
        for (int it = ft; it < (dead ? 0 : np * pl.na); it += F2_NF) {
          const int g = wt_fdiv(it, pl.d_na);
          const int rem = it - g * pl.na;
          const int bi = wt_fdiv(rem, pl.d_nbw);
          const int bj = rem - bi * pl.nbw;
          const T* rp = reinterpret_cast<const T*>(reinterpret_cast<const char*>(rawb) + g * pl.raw_pb);
          const int i0 = 4 * bi, j0 = 4 * bj;
          float v4[4][4];
          if (vec && i0 + 3 < H) {
#pragma unroll
            for (int a = 0; a < 4; ++a) raw_vec4<T>(rp, i0 + a, j0, W, v4[a]);
          } else {
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
              for (int e = 0; e < 4; ++e) v4[a][e] = raw_at<T>(rp, i0 + a, j0 + e, H, W);
          }
          // float32 input plane (interior only; 16-byte aligned rows)
          float* xd = sm + xo + g * XB.plane + (i0 + R) * XB.stride + j0 + 4;
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            if (i0 + a < H) {
              float* row = xd + a * XB.stride;
              if (j0 + 3 < W) {
                *reinterpret_cast<float4*>(row) = make_float4(v4[a][0], v4[a][1], v4[a][2], v4[a][3]);
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (j0 + e < W) row[e] = v4[a][e];
              }
            }
          }
          // level 1: four 2x2 butterflies; level 2 from their low-pass values
          float ll[2][2];
#pragma unroll
          for (int pu = 0; pu < 2; ++pu) {
            float o[2][4];
#pragma unroll
            for (int qv = 0; qv < 2; ++qv) {
              butterfly4(v4[2 * pu][2 * qv], v4[2 * pu][2 * qv + 1], v4[2 * pu + 1][2 * qv],
                         v4[2 * pu + 1][2 * qv + 1], o[qv]);
              ll[pu][qv] = o[qv][0];
            }
            const int p = 2 * bi + pu, q = 2 * bj;
            if (p < pl.Hs[1]) {
              float* d = sm + f2_at(B1, g, 0, p, q, R);
              if ((R & 1) == 0 && q + 1 < pl.Ws[1]) {
#pragma unroll
                for (int b = 0; b < 4; ++b) *reinterpret_cast<float2*>(d + b * B1.band) = make_float2(o[0][b], o[1][b]);
              } else {
#pragma unroll
                for (int qv = 0; qv < 2; ++qv)
                  if (q + qv < pl.Ws[1]) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) d[b * B1.band + qv] = o[qv][b];
                  }
              }
            }
          }
          if (L >= 2) {
            float o2[4];
            butterfly4(ll[0][0], ll[0][1], ll[1][0], ll[1][1], o2);
            float* d = sm + f2_at(B2, g, 0, bi, bj, R);
#pragma unroll
            for (int b = 0; b < 4; ++b) d[b * B2.band] = o2[b];
          }
        }
      }
      named_bar(1, F2_NF);
      named_arrive(F2_BAR_B1READY, F2_NT);       // X, B1 and the weights of unit v are ready
      if (!dead && v + 2 < nu) issue_count(v + 2);  // the raw slot is consumed
      // (2) levels 3..L of the analysis.
      for (int l = 3; l <= (dead ? 0 : L); ++l) {
        const WtF2Buf S = pl.B[l - 1], D = pl.B[l];
        const int Hl = pl.Hs[l], Wl = pl.Ws[l], per = Hl * Wl;
        for (int it = ft; it < np * per; it += F2_NF) {
          const int g = it / per;
          const int rem = it - g * per;
          const int p = rem / Wl, q = rem - p * Wl;
          const float* s = sm + f2_at(S, g, 0, 2 * p, 2 * q, R);
          float o[4];
          butterfly4(s[0], s[1], s[S.stride], s[S.stride + 1], o);
          float* d = sm + f2_at(D, g, 0, p, q, R);
#pragma unroll
          for (int b = 0; b < 4; ++b) d[b * D.band] = o[b];
        }
        named_bar(1, F2_NF);
      }
      // (3) band convolutions of levels 2..L (Zc).
      if (!dead && L >= 2) {
        for (int it = ft; it < np * pl.nco; it += F2_NF) {
          const int g = it / pl.nco;
          int l, b, r, s;
          f2_coarse_strip(pl, it - g * pl.nco, l, b, r, s);
          float w[KK];
          f2_load_w<K>(wsl + (1 + 4 * (l - 1) + b) * pl.wb, w);
          float acc[F2_SAC][4];
#pragma unroll
          for (int o = 0; o < F2_SAC; ++o)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[o][j] = 0.f;
          const WtF2Buf& Bl = pl.B[l];
          f2_strip<K, F2_SAC>(sm + f2_win(Bl, g, b, r, s, F2_SAC), Bl.stride, w, acc);
          const WtF2Buf& Zl = pl.Z[l];
          float* zd = sm + Zl.off + g * Zl.plane + b * Zl.band + F2_SAC * r * Zl.stride + 4 * s;
#pragma unroll
          for (int o = 0; o < F2_SAC; ++o)
            *reinterpret_cast<float4*>(zd + o * Zl.stride) = make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]);
        }
        named_bar(1, F2_NF);
        // (4) synthesis cascade of levels L..2 into R1 (level-1 resolution):
        // rec_{l-1}[2p+u][2q+v] = sum_b sign_b(u, v) (Zc_l,b + [b = 0] rec_l)[p][q].
        for (int l = L; l >= 2; --l) {
          const int Hl = pl.Hs[l], Wl = pl.Ws[l], per = Hl * Wl;
          const WtF2Buf Zl = pl.Z[l];
          const WtF2Buf Rin = pl.RC[l];  // rec_l (l < L)
          WtF2Buf Rout = pl.RC[l - 1];
          if (l == 2) Rout.off += slot * pl.r1slot + pl.zo;  // R1 columns shifted like Z1
          const int Hd = pl.Hs[l - 1], Wd = pl.Ws[l - 1];
          for (int it = ft; it < np * per; it += F2_NF) {
            const int g = it / per;
            const int rem = it - g * per;
            const int p = rem / Wl, q = rem - p * Wl;
            const float* z = sm + f2_at(Zl, g, 0, p, q, 0);
            float z0 = z[0];
            if (l < L) z0 += sm[f2_at(Rin, g, 0, p, q, 0)];
            const float z1 = z[Zl.band], z2 = z[2 * Zl.band], z3 = z[3 * Zl.band];
            float c4[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
            add_parities(z0, z1, z2, z3, c4);
            float* d = sm + f2_at(Rout, g, 0, 2 * p, 2 * q, 0);
#pragma unroll
            for (int uu = 0; uu < 2; ++uu)
#pragma unroll
              for (int vv = 0; vv < 2; ++vv)
                if (2 * p + uu < Hd && 2 * q + vv < Wd) d[uu * Rout.stride + vv] = c4[uu][vv];
          }
          named_bar(1, F2_NF);
        }
      }
      named_arrive(F2_BAR_FREADY, F2_NT);  // R1 of unit v is ready
    }
    named_bar(F2_BAR_MID, F2_NT);  // the consumers' last arrival
    // Copies still in flight (only after a failed wait) land before exit.
    if (bulk) {
      if (issued0 > waited0) f2_wait(&rawfull[0], (uint32_t)waited0 & 1u, pl.wait_shift);
      if (issued1 > waited1) f2_wait(&rawfull[1], (uint32_t)waited1 & 1u, pl.wait_shift);
    } else {
      cp_async_wait_all();
    }
  } else {
    // ======================= consumer group =======================
    const int bt = tid - F2_NF;
    const WtF2Buf B1 = pl.B[1], Z1 = pl.Z[1], XB = pl.X;
    const size_t HW = (size_t)H * W;
    for (int v = 0; v < nu; ++v) {
      const int u = u0 + v;
      const int c = wt_fdiv(u, pl.d_G);
      const int n0 = (u - c * pl.G) * P;
      const int np = min(P, pl.N - n0);
      const int slot = v & 1;
      const float* wsl = sm + pl.w_off + slot * pl.wslot;
      named_bar(F2_BAR_B1READY, F2_NT);  // X, B1 and the weights of unit v
      const bool dead = s_abort != 0;     // set before the producer's arrival: work is skipped
      // (a) level-1 band convolutions -> Z1.
      for (int k = bt; k < (dead ? 0 : np * pl.n1); k += F2_NB) {
        const F2Strip t = f2_l1_strip(pl, k);
        float w[KK];
        f2_load_w<K>(wsl + (1 + t.b) * pl.wb, w);
        float acc[F2_SA][4];
#pragma unroll
        for (int o = 0; o < F2_SA; ++o)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[o][j] = 0.f;
        f2_strip<K>(sm + f2_win(B1, t.g, t.b, t.r, t.s), B1.stride, w, acc);
        float* zd = sm + Z1.off + t.g * Z1.plane + t.b * Z1.band + F2_SA * t.r * Z1.stride + 4 * t.s + ZO;
#pragma unroll
        for (int o = 0; o < F2_SA; ++o) {
          float* zr = zd + o * Z1.stride;
          if constexpr (ZO == 0) {
            *reinterpret_cast<float4*>(zr) = make_float4(acc[o][0], acc[o][1], acc[o][2], acc[o][3]);
          } else {  // zo = 1: columns 4s+1 .. 4s+4
            zr[0] = acc[o][0];
            *reinterpret_cast<float2*>(zr + 1) = make_float2(acc[o][1], acc[o][2]);
            zr[3] = acc[o][3];
          }
        }
      }
      // R1 of unit v; this barrier also orders every consumer's Z1 writes
      // before the final strips read them.
      named_bar(F2_BAR_FREADY, F2_NT);
      named_arrive(F2_BAR_MID, F2_NT);  // B1 of unit v may be overwritten
      // (b) final strips: bias + level-1 synthesis of Z1 + R1, then the base
      // convolution accumulated on top, stored to HBM.
      if (!dead) {
        const float bias = (!ROT && b_base != nullptr) ? s_base[c] * b_base[c] : 0.f;
        float w[KK];
        f2_load_w<K>(wsl, w);
        const int xo = XB.off + slot * pl.xslot;
        const WtF2Buf R1 = pl.RC[1];
        const int r1o = R1.off + slot * pl.r1slot;
        for (int k = bt; k < np * pl.nf; k += F2_NB) {
          const F2Strip t = f2_final_strip(pl, k);
          const int c0 = 4 * t.s - SH;  // first output column of the strip
          const int qb = c0 >> 1;       // its level-1 column (floor)
          const float* zrow = sm + Z1.off + t.g * Z1.plane;
          const float* rrow = sm + r1o + t.g * R1.plane;
          float acc[F2_SA][4];
#pragma unroll
          for (int o = 0; o < F2_SA; ++o) {
            const int i = F2_SA * t.r + o;
            const int p = i >> 1;
            const float su = (i & 1) ? -1.f : 1.f;
            // level-1 synthesis: output column c0 + j takes level-1 column
            // qb + ((j + SH % 2) >> 1) with column parity (j + SH) & 1
            float zv[4][3], rv[3];
            if constexpr ((SH & 1) == 0) {
              const float* z = zrow + p * Z1.stride + qb + ZO;  // even: one 8-byte load per band
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const float2 t2 = *reinterpret_cast<const float2*>(z + b * Z1.band);
                zv[b][0] = t2.x;
                zv[b][1] = t2.y;
                zv[b][2] = 0.f;
              }
              float2 r2 = make_float2(0.f, 0.f);
              if (L >= 2) r2 = *reinterpret_cast<const float2*>(rrow + p * R1.stride + qb + ZO);
              rv[0] = r2.x;
              rv[1] = r2.y;
              rv[2] = 0.f;
            } else {
#pragma unroll
              for (int d = 0; d < 3; ++d) {
                const int q = max(qb + d, 0) + ZO;  // columns left of the plane feed only discarded outputs
#pragma unroll
                for (int b = 0; b < 4; ++b) zv[b][d] = zrow[b * Z1.band + p * Z1.stride + q];
                rv[d] = L >= 2 ? rrow[p * R1.stride + q] : 0.f;
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int d = (j + (SH & 1)) >> 1;
              const float a = fmaf(su, zv[1][d], zv[0][d] + rv[d]);
              const float bb = fmaf(su, zv[3][d], zv[2][d]);
              acc[o][j] = bias + ((((j + SH) & 1) == 0) ? a + bb : a - bb);
            }
          }
          f2_strip<K>(sm + xo + t.g * XB.plane + F2_SA * t.r * XB.stride + 4 * t.s, XB.stride, w, acc);
          T* plane = y + ((size_t)(n0 + t.g) * C + c) * HW;
#pragma unroll
          for (int o = 0; o < F2_SA; ++o) {
            const int i = F2_SA * t.r + o;
            if (i < H) {
              T* dst = plane + (size_t)i * W;
              if constexpr (SH == 0) {
                if (pl.out_vec && c0 + 4 <= W) {
                  stg_row<T, 4>(dst + c0, acc[o]);
                  continue;
                }
              } else if constexpr (SH == 2) {
                if (pl.out_vec && c0 >= 0 && c0 + 4 <= W) {  // two 2-element stores (c0 is even)
                  stg_row<T, 2>(dst + c0, acc[o]);
                  stg_row<T, 2>(dst + c0 + 2, acc[o] + 2);
                  continue;
                }
              }
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (c0 + j >= 0 && c0 + j < W) dst[c0 + j] = from_f32<T>(acc[o][j]);
            }
          }
        }
      }
      named_bar(2, F2_NB);  // Z1 is rewritten by the next unit
    }
  }
}

template <int K, typename T, bool ROT>
static cudaError_t launch_fwd2_t(const WtF2Plan& pl, const void* x, const float* w_base, const float* b_base,
                                 const float* w_sub, const float* s_base, const float* s_w, void* y,
                                 cudaStream_t stream) {
  auto kern = fwd2_kernel<K, T, ROT>;
  cudaError_t e = ensure_smem((const void*)kern, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  kern<<<pl.grid, F2_NT, pl.smem_bytes, stream>>>(pl, static_cast<const T*>(x), w_base, b_base, w_sub, s_base,
                                                  s_w, static_cast<T*>(y));
  return cudaGetLastError();
}

template <typename T, bool ROT>
static cudaError_t launch_fwd2_k(const WtF2Plan& pl, const void* x, const float* w_base, const float* b_base,
                                 const float* w_sub, const float* s_base, const float* s_w, void* y,
                                 cudaStream_t stream) {
  switch (pl.K) {
    case 3: return launch_fwd2_t<3, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 5: return launch_fwd2_t<5, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 7: return launch_fwd2_t<7, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    case 9: return launch_fwd2_t<9, T, ROT>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd2(const WtF2Plan& pl, bool rotate, const void* x, const float* w_base, const float* b_base,
                        const float* w_sub, const float* s_base, const float* s_w, void* y, cudaStream_t stream) {
  if (pl.dtype == 0)
    return rotate ? launch_fwd2_k<float, true>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_fwd2_k<float, false>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  if (pl.dtype == 1)
    return rotate ? launch_fwd2_k<__half, true>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                  : launch_fwd2_k<__half, false>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
  return rotate ? launch_fwd2_k<__nv_bfloat16, true>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream)
                : launch_fwd2_k<__nv_bfloat16, false>(pl, x, w_base, b_base, w_sub, s_base, s_w, y, stream);
}

// Resident CTAs per SM of the instantiation a plan launches.
int fwd2_ctas_per_sm(const WtF2Plan& pl) {
  const void* f = nullptr;
#define WT_F2_PICK(KV)                                                                                   \
  case KV:                                                                                               \
    f = pl.dtype == 0 ? (const void*)fwd2_kernel<KV, float, false>                                       \
                      : (pl.dtype == 1 ? (const void*)fwd2_kernel<KV, __half, false>                     \
                                       : (const void*)fwd2_kernel<KV, __nv_bfloat16, false>);            \
    break;
  switch (pl.K) {
    WT_F2_PICK(3)
    WT_F2_PICK(5)
    WT_F2_PICK(7)
    WT_F2_PICK(9)
    default: return 0;
  }
#undef WT_F2_PICK
  if (ensure_smem(f, pl.smem_bytes) != cudaSuccess) return 0;
  return occupancy(f, F2_NT, pl.smem_bytes);
}

unsigned int take_fwd2_faults() {
  unsigned int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd2_faults, sizeof(v)) != cudaSuccess) return 0;
  cudaMemcpyToSymbol(g_fwd2_faults, &z, sizeof(z));
  return v;
}

}  // namespace wt
