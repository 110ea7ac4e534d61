// pa_verify_inst.cu - the grouped balanced kernel on multi-token rows (a few
// new tokens per sequence, e.g. speculative verification), one translation
// unit per (cache type, q dtype): compiled with -DPA_INST_BF16={0,1} and
// -DPA_INST_FP8={0,1}; head_dim 128.
#include "pa_verify.cuh"

#ifndef PA_INST_BF16
#error "PA_INST_BF16 must be defined"
#endif
#ifndef PA_INST_FP8
#define PA_INST_FP8 0
#endif

#if PA_INST_FP8
#if PA_INST_BF16
#define PA_FN launch_multi_e4m3_bf16
#else
#define PA_FN launch_multi_e4m3_f16
#endif
#else
#if PA_INST_BF16
#define PA_FN launch_multi_bf16
#else
#define PA_FN launch_multi_f16
#endif
#endif

namespace pa {

cudaError_t PA_FN(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int nt,
                  int row_tiles, int head_group, dim3 grid, cudaStream_t st) {
  return launch_multi_rows<PA_INST_BF16 != 0, PA_INST_FP8 != 0>(tk, tv, a, nt, row_tiles,
                                                                head_group, grid, st);
}

}  // namespace pa
