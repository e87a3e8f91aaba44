// la_kernels_d64.cu -- instances of the decode kernels for head dim 64
// (LeanTile sizes 256, 128 tokens), query rows per kv head 1, 2, 4, 8 and 16, fp16 and bf16.
#include "la_kernel.cuh"

namespace la {

cudaError_t launch_decode_d64(int T, int grp, int dtype, const KParams& p, cudaStream_t st) {
  if (T == 256 && grp == 1)
    return dtype ? launch_decode_t<64, 256, 1, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 256, 1, __half>(p, st);
  if (T == 256 && grp == 2)
    return dtype ? launch_decode_t<64, 256, 2, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 256, 2, __half>(p, st);
  if (T == 256 && grp == 4)
    return dtype ? launch_decode_t<64, 256, 4, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 256, 4, __half>(p, st);
  if (T == 256 && grp == 8)
    return dtype ? launch_decode_t<64, 256, 8, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 256, 8, __half>(p, st);
  if (T == 256 && grp == 16)
    return dtype ? launch_decode_t<64, 256, 16, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 256, 16, __half>(p, st);
  if (T == 128 && grp == 1)
    return dtype ? launch_decode_t<64, 128, 1, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 128, 1, __half>(p, st);
  if (T == 128 && grp == 2)
    return dtype ? launch_decode_t<64, 128, 2, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 128, 2, __half>(p, st);
  if (T == 128 && grp == 4)
    return dtype ? launch_decode_t<64, 128, 4, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 128, 4, __half>(p, st);
  if (T == 128 && grp == 8)
    return dtype ? launch_decode_t<64, 128, 8, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 128, 8, __half>(p, st);
  if (T == 128 && grp == 16)
    return dtype ? launch_decode_t<64, 128, 16, __nv_bfloat16>(p, st)
                 : launch_decode_t<64, 128, 16, __half>(p, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine_d64(int grp, const CParams& p, cudaStream_t st) {
  switch (grp) {
    case 1: return launch_combine_t<64, 1>(p, st);
    case 2: return launch_combine_t<64, 2>(p, st);
    case 4: return launch_combine_t<64, 4>(p, st);
    case 8: return launch_combine_t<64, 8>(p, st);
    case 16: return launch_combine_t<64, 16>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t decode_capacity_d64(int T, int grp, int* per_sm) {
  if (T == 256 && grp == 1) return capacity_t<64, 256, 1>(per_sm);
  if (T == 256 && grp == 2) return capacity_t<64, 256, 2>(per_sm);
  if (T == 256 && grp == 4) return capacity_t<64, 256, 4>(per_sm);
  if (T == 256 && grp == 8) return capacity_t<64, 256, 8>(per_sm);
  if (T == 256 && grp == 16) return capacity_t<64, 256, 16>(per_sm);
  if (T == 128 && grp == 1) return capacity_t<64, 128, 1>(per_sm);
  if (T == 128 && grp == 2) return capacity_t<64, 128, 2>(per_sm);
  if (T == 128 && grp == 4) return capacity_t<64, 128, 4>(per_sm);
  if (T == 128 && grp == 8) return capacity_t<64, 128, 8>(per_sm);
  if (T == 128 && grp == 16) return capacity_t<64, 128, 16>(per_sm);
  return cudaErrorInvalidValue;
}

}  // namespace la
