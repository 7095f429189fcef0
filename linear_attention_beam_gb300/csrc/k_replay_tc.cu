// Fused shared-context replay on tcgen05 tensor cores: key width 128, and the
// shape checks and dispatch (the kernel is in replay_tc_impl.cuh; key width
// 256 is instantiated in k_replay_tc256.cu).
#include "replay_tc_impl.cuh"

namespace gdnbeam {

int launch_tc_replay_256(const ReplayArgs& a, cudaStream_t s);

bool tc_replay_supported(int dtype, int d_k, int d_v) {
  return dtype == GDNBEAM_BF16 && (d_k == 128 || d_k == 256) && d_v % VR == 0 && d_v <= 4 * VR;
}

int launch_tc_replay(const ReplayArgs& a, cudaStream_t s) {
  if (a.W_t <= 0) return GDNBEAM_OK;
  if (a.t > kMaxDepth || !tc_replay_supported(GDNBEAM_BF16, a.d_k, a.d_v))
    return launch_replay(GDNBEAM_BF16, a, s);
  return a.d_k == 128 ? launch_tc_replay_dk<128>(a, s) : launch_tc_replay_256(a, s);
}

}  // namespace gdnbeam
