// tc_gla.cu -- tcgen05 kernels (placeholder until the kernels land).
#include "tc.cuh"

namespace glacore {
namespace tc {

bool supported(const glacore_problem *, bool) { return false; }
int chunk_of(const glacore_problem *p) { return p->chunk_size ? p->chunk_size : 64; }
size_t workspace_bytes(const glacore_problem *, bool, bool) { return 0; }
cudaError_t fwd(const Prob &, const Docs &, const glacore_problem *, void *, float *, char *,
                cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t bwd(const Prob &, const Docs &, const glacore_problem *, const void *, const float *,
                void *, void *, void *, float *, float *, char *, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace tc
}  // namespace glacore
