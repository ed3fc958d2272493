// Fused WTConv2d backward: launch code and the instantiations (the kernel
// itself and its design are in wtconv_bwd_fused.cuh).  Only 8-row
// correlation tiles are built: with 4-row tiles (deep pyramids, small planes
// packed several per unit) the fused kernel measured no faster than the two
// separate passes on GB300 (7x7 and 14x14 fp16 layers of WTConvNeXt-T within
// 0.5 %, the 28x28 one at 4 levels 5 % slower), so those plans run the two
// passes.
#include "wtconv_bwd_fused.cuh"

namespace wt {

WT_BWF_INSTANTIATE(8)

static const void* bwf_pick(const WtBwPlan& pl, const WtFwdPlan& fp, int dtype) {
  if (fp.ftp != WT_TP / 2) return nullptr;  // half-height final tiles only
  return pl.tbr == 8 ? bwf_kernel_tr8(pl.K, dtype) : nullptr;
}

cudaError_t launch_bwd_fused(const WtBwPlan& pl, const WtFwdPlan& fp, const CUtensorMap& tmx, const CUtensorMap& tmd,
                             int dtype, const void* x, const void* dy, const float* w_base, const float* b_base,
                             const float* w_sub, const float* s_base, const float* s_w, void* dx, float* dw_base,
                             float* db_base, float* dw_sub, float* ds_base, float* ds_w, float* part,
                             cudaStream_t stream) {
  const void* f = bwf_pick(pl, fp, dtype);
  if (!f) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(f, pl.smem_bytes);
  if (e != cudaSuccess) return e;
  WtBwPlan plc = pl;
  WtFwdPlan fpc = fp;
  CUtensorMap mx = tmx, md = tmd;
  void* args[] = {(void*)&plc, (void*)&fpc, (void*)&mx, (void*)&md, (void*)&x, (void*)&dy, (void*)&w_base,
                  (void*)&w_sub, (void*)&s_base, (void*)&s_w, (void*)&dx, (void*)&part};
  e = cudaLaunchKernel(f, dim3((unsigned)pl.grid), dim3(WT_BW_THREADS), args, (size_t)pl.smem_bytes, stream);
  if (e != cudaSuccess) return e;
  return launch_bw_finalize(pl, part, w_base, b_base, w_sub, s_base, s_w, dw_base, db_base, dw_sub, ds_base, ds_w,
                            stream);
}

int bwf_ctas_per_sm(const WtBwPlan& pl, const WtFwdPlan& fp, int dtype) {
  const void* f = bwf_pick(pl, fp, dtype);
  if (!f) return 0;
  return occupancy(f, WT_BW_THREADS, pl.smem_bytes);
}

unsigned int take_bwf_faults() { return take_bwf_faults_tr8(); }

}  // namespace wt
