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
cudaError_t launch_build_units(const Docs &docs, int64_t plen, Unit *units, int64_t max_units,
                               cudaStream_t st);
// Units of a packed batch in launch order, longest first (counting sort by
// chunk count): long documents start in the first wave instead of the last.
cudaError_t launch_order_units(const Units &us, int64_t n, int32_t *order, cudaStream_t st);

// Scratch layout of the tcgen05 path (byte offsets into the workspace).
// Piece hand-off buffers (fp32): L [units,H,K,V] end state of each piece
// started from zero, D [units,H,K] exp(sum of g over the piece); Lr, Dr the
// same for the reverse pass (state gradient at the piece start).
struct TcLayout {
  int64_t plen, max_units, ckpt_slots;
  bool pieces, table;
  size_t off_units, off_order, off_L, off_D, off_Lr, off_Dr, off_dgp, off_bvec, off_ckpt, off_qt, off_kt, off_eng,
      off_egam, total;
};
// The backward resets the gate-gradient carry to the exact boundary term
// (S_end (.) dH_end) 1_V every CKPT_CHUNKS chunks (state written by pass A).
constexpr int CKPT_CHUNKS = 8;
TcLayout tc_layout(const glacore_problem *p, bool backward);

// Units of a launch under layout Lo: the table in the workspace (packed
// documents), implicit pieces of uniform rows, or one unit per document.
inline Units units_of(const Docs &docs, const TcLayout &Lo, char *ws) {
  Units us;
  us.docs = docs;
  us.table = (Lo.pieces && Lo.table) ? (const Unit *)(ws + Lo.off_units) : nullptr;
  us.plen = (Lo.pieces && !Lo.table) ? Lo.plen : 0;
  us.order = docs.start ? (const int32_t *)(ws + Lo.off_order) : nullptr;
  return us;
}

// Exact hand-off between pieces, folded into the consumer (no scan launch).
// Row c, columns v0 .. v0+N-1 of the state entering piece `piece` of a
// document whose first unit is u0:  S = h0 (or 0), then
//   S <- diag(D_q) S + L_q   for q = 0 .. piece-1.
template <int N>
__device__ __forceinline__ void piece_state_in(float (&S)[N], const float *h0row, const float *L,
                                               const float *D, int64_t u0, int piece, int64_t H,
                                               int64_t h, int c, int v0) {
#pragma unroll
  for (int i = 0; i < N; ++i) S[i] = h0row ? h0row[v0 + i] : 0.f;
  for (int q = 0; q < piece; ++q) {
    const int64_t uq = u0 + q;
    const float dq = D[(uq * H + h) * KD + c];
    const float4 *l = reinterpret_cast<const float4 *>(L + ((uq * H + h) * KD + c) * VD + v0);
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 x = l[i / 4];
      S[i] = dq * S[i] + x.x;
      S[i + 1] = dq * S[i + 1] + x.y;
      S[i + 2] = dq * S[i + 2] + x.z;
      S[i + 3] = dq * S[i + 3] + x.w;
    }
  }
}
// Row c, columns v0 .. v0+N-1 of the state gradient leaving piece `piece`
// (of npieces):  G = dht (or 0), then G <- diag(Dr_q) G + Lr_q for
// q = npieces-1 down to piece+1.
template <int N>
__device__ __forceinline__ void piece_grad_out(float (&G)[N], const float *dhtrow, const float *Lr,
                                               const float *Dr, int64_t u0, int piece, int npieces,
                                               int64_t H, int64_t h, int c, int v0) {
#pragma unroll
  for (int i = 0; i < N; ++i) G[i] = dhtrow ? dhtrow[v0 + i] : 0.f;
  for (int q = npieces - 1; q > piece; --q) {
    const int64_t uq = u0 + q;
    const float dq = Dr[(uq * H + h) * KD + c];
    const float4 *l = reinterpret_cast<const float4 *>(Lr + ((uq * H + h) * KD + c) * VD + v0);
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 x = l[i / 4];
      G[i] = dq * G[i] + x.x;
      G[i + 1] = dq * G[i + 1] + x.y;
      G[i + 2] = dq * G[i + 2] + x.z;
      G[i + 3] = dq * G[i + 3] + x.w;
    }
  }
}

// Launch of a kernel whose CTAs pair up along x in clusters of two.
template <typename... Params, typename... Args>
inline cudaError_t launch_pairs(void (*kernel)(Params...), dim3 grid, int smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(448, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct FwdMaps;
struct FwdArgs;
// The piece passes of the exact sequence split (tc_pieces.cu): the forward
// pass (local end state and total decay of every piece but the last of its
// document) and, when rm / ra are given, the reverse pass (local state
// gradient at the start of every piece but the first) in one launch.
cudaError_t launch_piece_states(const FwdMaps &fm, const FwdArgs &fa, const FwdMaps *rm, const FwdArgs *ra,
                                int64_t units, int64_t H, cudaStream_t st, bool rev_only = false);
// Local end state (from zero) and total decay of every document (forward),
// or, when dO is given, the local state gradient at every document's start
// (from zero at its end) and its total decay (reverse): the piece passes run
// with one unit per document.  L [n_docs,H,K,V], D [n_docs,H,K] fp32.
cudaError_t doc_states(const Prob &pr, const Docs &docs, const void *dO, float *L, float *D, cudaStream_t st);
cudaError_t fwd(const Prob &pr, const Docs &docs, const glacore_problem *p, void *o, float *ht,
                char *ws, cudaStream_t st);
cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO,
                const float *dht, void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws,
                cudaStream_t st);

}  // namespace tc
}  // namespace glacore
