// la_kernels_d128.cu -- instances of the decode kernels for head dim 128
// (LeanTile of 128 tokens), query-head groups 1, 2, 4 and 8, fp16 and bf16.
#include "la_kernel.cuh"

namespace la {

cudaError_t launch_decode_d128(int grp, int dtype, const KParams& p, cudaStream_t st) {
  switch (grp * 2 + dtype) {
    case 2: return launch_decode_t<128, 1, __half>(p, st);
    case 3: return launch_decode_t<128, 1, __nv_bfloat16>(p, st);
    case 4: return launch_decode_t<128, 2, __half>(p, st);
    case 5: return launch_decode_t<128, 2, __nv_bfloat16>(p, st);
    case 8: return launch_decode_t<128, 4, __half>(p, st);
    case 9: return launch_decode_t<128, 4, __nv_bfloat16>(p, st);
    case 16: return launch_decode_t<128, 8, __half>(p, st);
    case 17: return launch_decode_t<128, 8, __nv_bfloat16>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_d128(int grp, const CParams& p, cudaStream_t st) {
  switch (grp) {
    case 1: return launch_combine_t<128, 1>(p, st);
    case 2: return launch_combine_t<128, 2>(p, st);
    case 4: return launch_combine_t<128, 4>(p, st);
    case 8: return launch_combine_t<128, 8>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t decode_capacity_d128(int grp, int* per_sm) {
  switch (grp) {
    case 1: return capacity_t<128, 1>(per_sm);
    case 2: return capacity_t<128, 2>(per_sm);
    case 4: return capacity_t<128, 4>(per_sm);
    case 8: return capacity_t<128, 8>(per_sm);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
