// launch_ee.h -- the early-exit kernel whose clusters each walk one
// sequence's positions in order (verify_sample_ee.cu).
#pragma once

#include "launch.h"

namespace specv {

// One cluster of C CTAs per sequence, each row pair staged in shared memory;
// the draw at the first rejection reads nothing again.  ee_cluster: the
// cluster size the rows need (0: they do not fit).
int ee_cluster(long long nvec);
cudaError_t sample_ee_prepare();
cudaError_t launch_sample_ee(const VerifyArgs& a, int C, cudaStream_t stream);

}  // namespace specv
