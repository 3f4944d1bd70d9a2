// Temporary: tensor-core launchers not yet built.
#include "gla_internal.h"
namespace gla {
cudaError_t launch_prep(const gla_fwd_params&, const Plan&, void*, int*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_chunk_fwd(const gla_fwd_params&, const Plan&, void*, int, int*, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_seg_scan(const gla_fwd_params&, const Plan&, void*, int*, cudaStream_t) { return cudaErrorNotSupported; }
}
