// ssd_fused_tc.cu -- fused tcgen05/TMA path (not built yet: reports unsupported).
#include "ssd_internal.cuh"

namespace ssd {

bool fused_supports(const Problem &) { return false; }
size_t fused_workspace_bytes(const Problem &) { return kStatusBytes; }
cudaError_t fused_launch(const Problem &, void *, size_t, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace ssd
