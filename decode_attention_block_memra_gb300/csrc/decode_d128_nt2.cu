// Instantiations of the split-K decode kernel for head_dim 128, 2 n-tile(s) of
// 8 query rows per warp (all six K/V format pairs); split across translation
// units so they compile in parallel.
#include "decode_kernel.cuh"

namespace memra {

cudaError_t launch_decode_d128_nt2(int kf, int vf, const DecodeParams &p, dim3 grid, size_t smem, cudaStream_t st) {
  return dispatch_formats<128, 2>(kf, vf, p, grid, smem, st);
}

}  // namespace memra
