// tc_ssd.cuh -- tcgen05 kernels for Mamba-2 SSD: one log-decay per head and
// token, q / k (C / B) shared by a group of heads, bf16 inputs, K = 128
// state channels, V = 64 head dims, chunk C = 64.
//
// Chunk formulas (FLAT blog, trainstation-project.github.io/blog/flat:
// "Mamba-2" for the scalar per-head decay and its C x C decay matrix, taken
// in log space; "Linear Attention / Forward Recurrence" for the chunkwise
// form; "Backward Recurrence" for the reverse walk):
//
//   G_t  = inclusive prefix sum of g over the chunk (one value per token)
//   Gam  = G at the chunk's last token
//   D    = exp(G_t - G_s) for s <= t, else 0          (C x C, per head)
//   P    = scale (q k^T) (.) D
//   O    = scale diag(exp(G)) q S + P v
//   S   <- exp(Gam) S + k^T diag(exp(Gam - G)) v
//
// Unlike the per-channel GLA kernels, no factor is split into exp(G_t) and
// exp(-G_s): every exponent is a difference G_t - G_s with s <= t, or
// Gam - G_s, or G_t, so with g <= 0 (Mamba-2's dt * A) every factor lies in
// (0, 1] and any decay strength is exact.  q k^T is computed once per chunk
// and then decayed with this head's D.
#pragma once

#include "tc_common.cuh"

namespace glacore {
namespace ssd {

constexpr int C = 64;
constexpr int KD = 128;  // state channels (N)
constexpr int VD = 64;   // head dim (P)

// True when these kernels run the SSD problem: bf16, K = 128, V = 64, any
// head grouping, q / k / v token strides TMA can address, chunk 0 or 64.
bool supported(const glacore_problem *p);
// Scratch of the SSD kernels (launch order of packed documents; the
// backward's fp32 dq / dk accumulators and per-token gate-gradient terms).
size_t workspace_bytes(const glacore_problem *p, bool backward);
cudaError_t fwd(const Prob &pr, const Docs &docs, const glacore_problem *p, void *o, float *ht, char *ws,
                cudaStream_t st);
cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO, const float *dht,
                void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws, cudaStream_t st);

}  // namespace ssd
}  // namespace glacore
