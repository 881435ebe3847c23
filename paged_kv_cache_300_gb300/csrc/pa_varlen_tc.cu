// bf16 varlen attention on tcgen05 tensor cores (in progress).
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

int varlen_bf16_launch(const VarlenArgs &, const CUtensorMap &, const CUtensorMap &,
                       const CUtensorMap &, cudaStream_t)
{
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
