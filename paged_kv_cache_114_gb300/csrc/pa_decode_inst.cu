// pa_decode_inst.cu - one decode instantiation per (cache type, dtype, head_dim).
// Compiled once per combination with -DPA_INST_BF16={0,1} -DPA_INST_D={64,128,256}
// and -DPA_INST_FP8={0,1} (E4M3 caches, head_dim 128 or 256) so the variants
// build in parallel.
#include "pa_decode_grouped.cuh"

#ifndef PA_INST_BF16
#error "PA_INST_BF16 must be defined"
#endif
#ifndef PA_INST_D
#error "PA_INST_D must be defined"
#endif
#ifndef PA_INST_FP8
#define PA_INST_FP8 0
#endif

#define PA_CAT3(a, b, c) a##b##c
#if PA_INST_FP8
#define PA_NAME(dt, d) PA_CAT3(launch_decode_e4m3_, dt, d)
#else
#define PA_NAME(dt, d) PA_CAT3(launch_decode_, dt, d)
#endif
#if PA_INST_BF16
#define PA_FN PA_NAME(bf16_, PA_INST_D)
#else
#define PA_FN PA_NAME(f16_, PA_INST_D)
#endif

namespace pa {

cudaError_t PA_FN(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int group_tiles,
                  int head_group, dim3 grid, int kernel, cudaStream_t st) {
  constexpr bool kBf16 = PA_INST_BF16 != 0;
  constexpr bool kFp8 = PA_INST_FP8 != 0;
  static_assert(!kFp8 || PA_INST_D >= 128, "E4M3 caches need head_dim 128 or 256");
  if (kernel == kGroupedRanges) {
    if (group_tiles == 1)
      return launch_grouped_tiles<kBf16, PA_INST_D, 1, kFp8>(tk, tv, a, head_group, grid, st);
    if (group_tiles == 2)
      return launch_grouped_tiles<kBf16, PA_INST_D, 2, kFp8>(tk, tv, a, head_group, grid, st);
    return cudaErrorInvalidValue;
  }
  return launch_decode_dispatch<kBf16, PA_INST_D, kFp8>(tk, tv, a, group_tiles, grid,
                                                        kernel == kPerWarpRanges, st);
}

}  // namespace pa
