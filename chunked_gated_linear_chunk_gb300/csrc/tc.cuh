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

// Chunk length of the tcgen05 kernels and their head dims.
constexpr int C = 64;
constexpr int KD = 128;
constexpr int VD = 128;

// exact sequence split (tc_pieces.cu)
int64_t piece_len(const glacore_problem *p, bool backward);
int64_t max_units_of(const glacore_problem *p, int64_t plen);
cudaError_t launch_build_units(const Docs &docs, int64_t plen, Unit *units, int64_t *ubase,
                               int64_t max_units, cudaStream_t st);
cudaError_t launch_fwd_scan(const Docs &docs, const int64_t *ubase, int64_t H, const float *h0,
                            const float *L, const float *D, float *sin, cudaStream_t st);
cudaError_t launch_rev_scan(const Docs &docs, const int64_t *ubase, int64_t H, const float *dht,
                            const float *Lr, const float *D, float *dhend, cudaStream_t st);

// Scratch layout of the tcgen05 path (byte offsets into the workspace).
struct TcLayout {
  int64_t plen, max_units, ckpt_slots;
  bool pieces;
  size_t off_units, off_ubase, off_L, off_D, off_sin, off_dhend, off_dgp, off_bvec, off_ckpt, total;
};
// The backward resets the gate-gradient carry to the exact boundary term
// (S_end (.) dH_end) 1_V every CKPT_CHUNKS chunks (state written by pass A).
constexpr int CKPT_CHUNKS = 8;
TcLayout tc_layout(const glacore_problem *p, bool backward);

cudaError_t fwd(const Prob &pr, const Docs &docs, const glacore_problem *p, void *o, float *ht,
                char *ws, cudaStream_t st);
cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO,
                const float *dht, void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws,
                cudaStream_t st);

}  // namespace tc
}  // namespace glacore
