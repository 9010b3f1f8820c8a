// linear_tc.cu -- tensor-core (tcgen05) path of the linear memory update.
#include "common.cuh"
#include "kernels.h"

namespace atlas {

bool linear_tc_supported(const LinArgs&) { return false; }

int linear_tc_launch(const LinArgs&, int, int*, cudaStream_t) { return ATLAS_ERR_UNSUPPORTED; }

}  // namespace atlas
