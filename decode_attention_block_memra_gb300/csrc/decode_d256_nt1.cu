// Instantiations of the split-K decode kernel for head_dim 256, 1 n-tile(s) of
// 8 query rows per warp (all six K/V format pairs); split across translation
// units so they compile in parallel.
#include "decode_kernel.cuh"

namespace memra {

cudaError_t launch_decode_d256_nt1(int kf, int vf, const DecodeParams &p, dim3 grid, size_t smem, cudaStream_t st) {
  return dispatch_formats<256, 1>(kf, vf, p, grid, smem, st);
}

}  // namespace memra
