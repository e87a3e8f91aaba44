// la_kernels_d64_hp2.cu -- instances of the decode kernel for head dim 64 with
// units of 2 kv heads (token-major and paged caches: 256-byte pieces per token
// row instead of 128), 128 tokens of each head per tile, query-head groups 1, 2, 4
// and 8, fp16 and bf16.
#include "la_kernel.cuh"

namespace la {

cudaError_t launch_decode_d64_hp2(int T, int grp, int dtype, const KParams& p, cudaStream_t st) {
  if (T == 128 && grp == 1)
    return dtype ? launch_decode_t<64, 128, 1, __nv_bfloat16, 2>(p, st)
                 : launch_decode_t<64, 128, 1, __half, 2>(p, st);
  if (T == 128 && grp == 2)
    return dtype ? launch_decode_t<64, 128, 2, __nv_bfloat16, 2>(p, st)
                 : launch_decode_t<64, 128, 2, __half, 2>(p, st);
  if (T == 128 && grp == 4)
    return dtype ? launch_decode_t<64, 128, 4, __nv_bfloat16, 2>(p, st)
                 : launch_decode_t<64, 128, 4, __half, 2>(p, st);
  if (T == 128 && grp == 8)
    return dtype ? launch_decode_t<64, 128, 8, __nv_bfloat16, 2>(p, st)
                 : launch_decode_t<64, 128, 8, __half, 2>(p, st);
  return cudaErrorInvalidValue;
}

cudaError_t decode_capacity_d64_hp2(int T, int grp, int* per_sm) {
  if (T == 128 && grp == 1) return capacity_t<64, 128, 1, 2>(per_sm);
  if (T == 128 && grp == 2) return capacity_t<64, 128, 2, 2>(per_sm);
  if (T == 128 && grp == 4) return capacity_t<64, 128, 4, 2>(per_sm);
  if (T == 128 && grp == 8) return capacity_t<64, 128, 8, 2>(per_sm);
  return cudaErrorInvalidValue;
}

}  // namespace la
