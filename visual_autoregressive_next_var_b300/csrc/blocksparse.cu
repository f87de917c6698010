// Block-sparse cross-scale attention (placeholder launcher until the kernel lands).
#include "internal.h"

namespace varattn {

int launch_attn_blocksparse(const StepGeom&, const int32_t*, int, int, const void*, const void*,
                            const void*, const var_block_mask*, void*, cudaStream_t)
{
    return VAR_ERR_UNSUPPORTED;
}

}  // namespace varattn
