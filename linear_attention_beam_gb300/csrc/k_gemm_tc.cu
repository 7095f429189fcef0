// tcgen05 tensor-core GEMMs (placeholder until the kernels land).
#include "common.cuh"
#include "launchers.h"

namespace gdnbeam {

bool tc_gemm_supported(const gdnbeam_config&) { return false; }
int launch_tc_project(const gdnbeam_config&, int, const void*, const void*, void*, void*, void*,
                      float*, float*, const gdnbeam_dumps*, cudaStream_t) {
  return GDNBEAM_EUNSUPPORTED;
}
size_t tc_logits_scratch_bytes(const gdnbeam_config&, int) { return 0; }
int launch_tc_logits(const gdnbeam_config&, int, const void*, const void*, void*, float*, void*,
                     const gdnbeam_dumps*, cudaStream_t) {
  return GDNBEAM_EUNSUPPORTED;
}
bool tc_replay_supported(int, int, int) { return false; }
int launch_tc_replay(const ReplayArgs&, cudaStream_t) { return GDNBEAM_EUNSUPPORTED; }

}  // namespace gdnbeam
