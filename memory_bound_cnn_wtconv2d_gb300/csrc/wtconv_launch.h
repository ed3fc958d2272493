// Internal launchers of libwtconv (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "wtconv_plan.h"

namespace wt {

// Forward pass (rotate = false) or input-gradient pass (rotate = true, no bias).
// tmx describes x for the TMA path (used when pl.use_tma).
cudaError_t launch_fwd(const WtFwdPlan& pl, const CUtensorMap& tmx, int dtype, bool rotate, const void* x,
                       const float* w_base, const float* b_base, const float* w_sub, const float* s_base,
                       const float* s_w, void* y, cudaStream_t stream);

// The same passes for planes too large for one CTA, tile by tile with a halo
// (pl.win = 1); tmx describes x for the box copies (pl.win_load = 1 or 2).
cudaError_t launch_fwd_win(const WtFwdPlan& pl, const CUtensorMap& tmx, int dtype, bool rotate, const void* x,
                           const float* w_base, const float* b_base, const float* w_sub, const float* s_base,
                           const float* s_w, void* y, cudaStream_t stream);

// Number of bounded in-kernel waits that gave up since the last call
// (reads and clears a device counter; synchronises the device).
unsigned int take_fwd_faults();
unsigned int take_win_faults();
unsigned int take_bww_faults();
unsigned int take_bwf_faults();
unsigned int take_bw_faults();

// Parameter gradients: correlation kernel into `part`, then the finalize kernel.
cudaError_t launch_bwd_weight(const WtBwPlan& pl, const CUtensorMap& tmx, const CUtensorMap& tmd, int dtype,
                              const void* x, const void* dy,
                              const float* w_base, const float* b_base, const float* w_sub,
                              const float* s_base, const float* s_w, float* dw_base, float* db_base,
                              float* dw_sub, float* ds_base, float* ds_w, float* part,
                              cudaStream_t stream);

// The finalize alone: adds each channel's records in CTA order and unfolds
// the scales (shared by the whole-plane and the windowed gradient passes).
cudaError_t launch_bw_finalize(const WtBwPlan& pl, const float* part, const float* w_base, const float* b_base,
                               const float* w_sub, const float* s_base, const float* s_w, float* dw_base,
                               float* db_base, float* dw_sub, float* ds_base, float* ds_w, cudaStream_t stream);

// Parameter gradients for planes beyond one CTA, tile by tile with a halo on
// x (pl.win = 1); tmx / tmd describe x and dy for the box copies.
cudaError_t launch_bwd_weight_win(const WtBwPlan& pl, const CUtensorMap& tmx, const CUtensorMap& tmd, int dtype,
                                  const void* x, const void* dy, const float* w_base, const float* b_base,
                                  const float* w_sub, const float* s_base, const float* s_w, float* dw_base,
                                  float* db_base, float* dw_sub, float* ds_base, float* ds_w, float* part,
                                  cudaStream_t stream);

// Fused backward: input gradient (into dx) and parameter gradients (records
// into `part`, then the finalize) from one kernel over x and dy.
cudaError_t launch_bwd_fused(const WtBwPlan& pl, const WtFwdPlan& fp, const CUtensorMap& tmx, const CUtensorMap& tmd,
                             int dtype, const void* x, const void* dy, const float* w_base, const float* b_base,
                             const float* w_sub, const float* s_base, const float* s_w, void* dx, float* dw_base,
                             float* db_base, float* dw_sub, float* ds_base, float* ds_w, float* part,
                             cudaStream_t stream);
int bwf_ctas_per_sm(const WtBwPlan& pl, const WtFwdPlan& fp, int dtype);

// Resident parameter-gradient CTAs per SM for a plan, from the runtime's
// occupancy calculator (0 when it cannot tell).
int bw_ctas_per_sm(const WtBwPlan& pl, int dtype);
// Registers per thread of the whole-plane gradient kernel with 4-row tiles,
// mi (1 or 2) tiles per thread, read once from the runtime (0 when it cannot tell).
int bw_regs(int k, int mi, int dtype);
int bw_win_ctas_per_sm(const WtBwPlan& pl, int dtype);
// Registers per thread of the windowed gradient kernel for (k, tile rows,
// dtype), read once from the runtime (0 when it cannot tell).
int bw_win_regs(int k, int tbr, int dtype);
// The same for the whole-plane forward kernel (k, dtype).
int fwd_regs(int k, int dtype);

// Coarse-level split (layers whose tile window does not fit one CTA):
//   launch_lowpass: ll = block sums of x over 2^s x 2^s blocks (float32,
//     planes x ceil(H / 2^s) x ceil(W / 2^s));
//   launch_add_carry: y[i][j] += c[i >> s][j >> s] on every plane;
//   launch_scale: out[i] = f * in[i] (in may equal out).
cudaError_t launch_lowpass(int dtype, const void* x, float* ll, long long planes, int H, int W, int s,
                           cudaStream_t stream);
cudaError_t launch_add_carry(int dtype, void* y, const float* c, long long planes, int H, int W, int s,
                             cudaStream_t stream);
cudaError_t launch_scale(const float* in, float* out, int n, float f, cudaStream_t stream);

// Sets the thread-local message returned by wtconv_last_error().
void set_last_error(const char* msg);

// Host-side caches, per device, of what every call would otherwise ask the
// runtime again (each a few microseconds):
//   ensure_smem: raises kernel f's opt-in dynamic shared-memory limit to at
//     least `bytes` (one cudaFuncSetAttribute per new maximum);
//   occupancy: resident CTAs per SM of f at `threads` threads and `smem`
//     dynamic bytes (after ensure_smem), 0 if the runtime cannot tell;
//   sm_count: the current device's SM count.
cudaError_t ensure_smem(const void* f, int bytes);
int occupancy(const void* f, int threads, int smem);
int sm_count();

}  // namespace wt
