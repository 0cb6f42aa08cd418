// tc_pieces.cu -- exact sequence split for the tensor-core kernels.
//
// A document whose (document x head) count is too small to fill the GPU is
// cut into pieces of P tokens (P a multiple of the chunk length) that run in
// parallel.  The hand-off between pieces is exact (JLA product page,
// karlex.ai/jla: "our split is exact", unlike starting every piece from
// zero): the recurrence is linear in the state, so with
//   L_p = end state of piece p started from zero,  D_p = exp(sum of g over p)
// the state entering piece p is
//   S_in[0] = h0,   S_in[p] = diag(D_{p-1}) S_in[p-1] + L_{p-1},
// and in reverse time, with Lr_p the state gradient at the start of piece p
// from its own outputs started from zero at its end,
//   dH_end[last] = dht,   dH_end[p] = diag(D_{p+1}) dH_end[p+1] + Lr_{p+1}.
// The consumers fold these recurrences over the earlier (later) pieces of
// their document when they start (piece_state_in / piece_grad_out in
// tc.cuh); the local states come from state-only modes of the forward and
// reverse kernels.  This file builds the unit table of packed documents and
// sizes the workspace.
#include "tc.cuh"

namespace glacore {
namespace tc {

// One CTA: packed documents -> pieces of `plen` tokens, in document order
// (the pieces of one document are consecutive units); units past the last
// piece are empty.
__global__ void __launch_bounds__(1024)
    build_units_kernel(Docs docs, int64_t plen, Unit *units, int64_t max_units) {
  __shared__ int64_t wbuf[32];
  __shared__ int64_t base_of_chunk;
  int64_t off = 0;
  for (int64_t base = 0; base < docs.n; base += blockDim.x) {
    const int64_t d = base + threadIdx.x;
    int64_t np = 0, s = 0, e = 0;
    if (d < docs.n) {
      docs.range(d, s, e);
      np = (e - s + plen - 1) / plen;
    }
    int64_t tot;
    const int64_t ex = block_excl_scan(np, wbuf, tot);
    for (int64_t p = 0; p < np; ++p) {
      const int64_t u = off + ex + p;
      if (u >= max_units) break;
      Unit r;
      r.start = s + p * plen;
      r.end = min(e, r.start + plen);
      r.doc = (int32_t)d;
      r.piece = (int32_t)p;
      r.npieces = (int32_t)np;
      r.pad = 0;
      units[u] = r;
    }
    off += tot;
  }
  if (threadIdx.x == 0) base_of_chunk = off;
  __syncthreads();
  for (int64_t u = base_of_chunk + threadIdx.x; u < max_units; u += blockDim.x) {
    Unit r;
    r.start = r.end = 0;
    r.doc = r.piece = r.pad = 0;
    r.npieces = 1;
    units[u] = r;
  }
}

cudaError_t launch_build_units(const Docs &docs, int64_t plen, Unit *units, int64_t max_units,
                               cudaStream_t st) {
  build_units_kernel<<<1, 1024, 0, st>>>(docs, plen, units, max_units);
  mark_launch("build_units", st);
  return cudaGetLastError();
}

// Piece length: split documents only when (documents x heads x CTAs per
// unit) leaves most of the GPU's SMs idle, and then into about as many
// pieces as make one wave.
int64_t piece_len(const glacore_problem *p, bool backward) {
  const int64_t sms = 148;  // one CTA per SM (GB300: 152 SMs)
  const int64_t per_unit = backward ? 1 : 2;
  const int64_t units = p->n_seqs * p->H * per_unit;
  const int64_t never = (int64_t)1 << 40;
  if (units <= 0 || units * 4 >= sms * 3) return never;
  const int64_t want = sms / units;  // pieces per document
  if (want < 2) return never;
  const int64_t avg = (p->B * p->T + p->n_seqs - 1) / p->n_seqs;
  int64_t plen = (avg + want - 1) / want;
  plen = ((plen + C - 1) / C) * C;
  if (plen < 4 * C) plen = 4 * C;
  return plen >= avg ? never : plen;
}

int64_t max_units_of(const glacore_problem *p, int64_t plen) {
  if (plen >= ((int64_t)1 << 40)) return p->n_seqs;
  if (!p->segment_ids) return p->B * ((p->T + plen - 1) / plen);
  return p->n_seqs + (p->B * p->T + plen - 1) / plen;
}

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

TcLayout tc_layout(const glacore_problem *p, bool backward) {
  TcLayout L;
  L.plen = piece_len(p, backward);
  L.pieces = L.plen < ((int64_t)1 << 40);
  L.table = L.pieces && p->segment_ids != nullptr;
  L.max_units = max_units_of(p, L.plen);
  const size_t mu = (size_t)L.max_units, H = (size_t)p->H;
  const size_t state = (size_t)KD * VD * sizeof(float);
  size_t off = 0;
  L.off_units = L.off_L = L.off_D = L.off_Lr = L.off_Dr = L.off_dgp = L.off_bvec = L.off_ckpt = 0;
  L.off_qt = L.off_kt = 0;
  // chunks of all documents (upper bound) -> checkpoint slots
  const int64_t chunks = p->segment_ids ? (p->B * p->T + C - 1) / C + p->n_seqs
                                        : p->B * ((p->T + C - 1) / C);
  L.ckpt_slots = chunks / CKPT_CHUNKS + 1;
  if (L.pieces) {
    if (L.table) {
      L.off_units = off;
      off = al256(off + mu * sizeof(Unit));
    }
    L.off_L = off;
    off = al256(off + mu * H * state);
    L.off_D = off;
    off = al256(off + mu * H * KD * sizeof(float));
    if (backward) {
      L.off_Lr = off;
      off = al256(off + mu * H * state);
      L.off_Dr = off;
      off = al256(off + mu * H * KD * sizeof(float));
    }
  }
  if (backward) {
    // q (.) dq partials per chunk slot (global chunk index), channel-major
    L.off_dgp = off;
    off = al256(off + (size_t)chunks * H * KD * C * sizeof(float));
    L.off_bvec = off;
    off = al256(off + mu * H * KD * sizeof(float));
    L.off_ckpt = off;
    off = al256(off + (size_t)L.ckpt_slots * H * state);
    // gated operands of pass B, written by pass A: qt = scale q exp(G), kt = k exp(-G)
    L.off_qt = off;
    off = al256(off + (size_t)p->B * p->T * H * KD * 2);
    L.off_kt = off;
    off = al256(off + (size_t)p->B * p->T * H * KD * 2);
  }
  L.total = off;
  return L;
}

}  // namespace tc
}  // namespace glacore
