// Instantiations of the split-K decode kernel for head_dim 128 (all six K/V
// format pairs); one translation unit per head_dim so they compile in parallel.
#include "decode_kernel.cuh"

namespace memra {

cudaError_t launch_decode_d128(int kf, int vf, const DecodeParams &p, dim3 grid, size_t smem, cudaStream_t st) {
  return dispatch_formats<128>(kf, vf, p, grid, smem, st);
}

}  // namespace memra
