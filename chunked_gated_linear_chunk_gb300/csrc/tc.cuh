// tc.cuh -- the tensor-core (tcgen05 / TMEM / TMA) path for bf16 inputs.
#pragma once

#include "internal.cuh"

namespace glacore {
namespace tc {

// True when the tcgen05 kernels cover this problem (bf16, K = V = 128,
// per-key-channel gate with one q/k head per value head).
bool supported(const glacore_problem *p, bool head_gate, bool backward);
// Chunk length used by the tcgen05 kernels for this problem.
int chunk_of(const glacore_problem *p);
// Scratch the tcgen05 path needs (state workspace of the backward).
size_t workspace_bytes(const glacore_problem *p, bool head_gate, bool backward);

cudaError_t fwd(const Prob &pr, const Docs &docs, const glacore_problem *p, void *o, float *ht,
                char *ws, cudaStream_t st);
cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO,
                const float *dht, void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws,
                cudaStream_t st);

}  // namespace tc
}  // namespace glacore
