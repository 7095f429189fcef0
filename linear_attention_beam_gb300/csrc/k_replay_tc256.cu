// Fused shared-context replay on tcgen05 tensor cores, key width 256 (its own
// translation unit so the two widths compile in parallel).
#include "replay_tc_impl.cuh"

namespace gdnbeam {

int launch_tc_replay_256(const ReplayArgs& a, cudaStream_t s) { return launch_tc_replay_dk<256>(a, s); }

}  // namespace gdnbeam
