// Tensor-core (tcgen05) chunked causal forward: not built yet.
#include "la_common.cuh"
#include "la_internal.h"

namespace la {

la_status causal_tc(const Problem &) { return LA_ERR_UNSUPPORTED; }

la_status tc_causal_read_status(cudaStream_t, unsigned *bits)
{
    *bits = 0;
    return LA_OK;
}

}  // namespace la
