// la_kernels_wide.cu -- instances of the tcgen05 decode kernel for units of
// up to 128 query rows (head dims 64, 80, 96 and 128, 128-token LeanTiles) and
// up to 64 rows at head dim 256 (64-token LeanTiles), fp16 and bf16, and the
// fixed-split merge for their records.
#include "la_wide.cuh"

namespace la {

bool wide_supported(int d) { return d == 64 || d == 80 || d == 96 || d == 128 || d == 256; }

int wide_tile(int d) { return d == 256 ? WCfg<256>::T : kWideTile; }

int wide_max_rows(int d) { return d == 256 ? WCfg<256>::MAX_ROWS : kWideRows; }

cudaError_t launch_wide(int d, int dtype, const KParams& p, cudaStream_t st) {
  switch (d) {
    case 64: return dtype ? launch_wide_t<64, __nv_bfloat16>(p, st) : launch_wide_t<64, __half>(p, st);
    case 80: return dtype ? launch_wide_t<80, __nv_bfloat16>(p, st) : launch_wide_t<80, __half>(p, st);
    case 96: return dtype ? launch_wide_t<96, __nv_bfloat16>(p, st) : launch_wide_t<96, __half>(p, st);
    case 128: return dtype ? launch_wide_t<128, __nv_bfloat16>(p, st) : launch_wide_t<128, __half>(p, st);
    case 256: return dtype ? launch_wide_t<256, __nv_bfloat16>(p, st) : launch_wide_t<256, __half>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t wide_capacity(int d, int* per_sm) {
  switch (d) {
    case 64: return wide_capacity_t<64>(per_sm);
    case 80: return wide_capacity_t<80>(per_sm);
    case 96: return wide_capacity_t<96>(per_sm);
    case 128: return wide_capacity_t<128>(per_sm);
    case 256: return wide_capacity_t<256>(per_sm);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_combine_wide(int d, const CParams& p, cudaStream_t st) {
  switch (d) {
    case 64: return launch_wide_combine_t<64>(p, st);
    case 80: return launch_wide_combine_t<80>(p, st);
    case 96: return launch_wide_combine_t<96>(p, st);
    case 128: return launch_wide_combine_t<128>(p, st);
    case 256: return launch_wide_combine_t<256>(p, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace la
