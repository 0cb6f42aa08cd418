// tc_gla.cu -- host side of the tcgen05 forward (kernel body in tc_gla_fwd.cuh).
#include <stdio.h>

#include <string.h>

#include "tc_gla_fwd.cuh"

namespace glacore {
namespace tc {

// HG: one gate per head (SSD); otherwise one per key channel
template <bool HG>
__global__ void __launch_bounds__(448, 1)
    gla_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs a) {
  gla_fwd_body<HG>(maps, a, blockIdx.x);
}

// =========================================================================
// host side
// =========================================================================

// True when the tcgen05 kernels cover this GLA problem (bf16, K = V = 128,
// any head sharing H % Hqk == 0; a token stride of q / k / v that TMA can
// address: a multiple of 16 bytes).
static bool strides_ok(const glacore_problem *p) {
  return (p->q_stride % 8) == 0 && (p->k_stride % 8) == 0 && (p->v_stride % 8) == 0;
}
bool supported(const glacore_problem *p, bool head_gate, bool) {
  if (head_gate) return false;
  return p->dtype == GLACORE_BF16 && p->K == KD && p->V == VD && p->H % p->Hqk == 0 && strides_ok(p) &&
         (p->chunk_size == 0 || p->chunk_size == 64) && p->B * p->T < ((int64_t)1 << 31) &&
         // one-dimensional grids of 2 x units x heads CTAs (units <= documents + pieces)
         4 * p->B * p->T * p->H < ((int64_t)1 << 31);
}
int chunk_of(const glacore_problem *) { return C; }
size_t workspace_bytes(const glacore_problem *p, bool, bool backward) {
  return tc_layout(p, backward).total;
}

cudaError_t fwd(const Prob &pr, const Docs &docs, const glacore_problem *p, void *o, float *ht,
                char *ws, cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
  if (const cudaError_t be = bind_context()) return be;
  const TcLayout Lo = tc_layout(p, false);
  FwdMaps maps;
  const int64_t BT = pr.BT;
  memset(&maps, 0, sizeof(maps));
  if (!make_map(&maps.q, pr.q, true, KD, pr.Hqk, BT, 64, pr.qs) ||
      !make_map(&maps.k, pr.k, true, KD, pr.Hqk, BT, 64, pr.ks) ||
      !make_map(&maps.v, pr.v, true, pr.V, pr.H, BT, 64, pr.vs) ||
      (!pr.gate_head && !make_map(&maps.g, pr.g, false, KD, pr.H, BT, 32)))
    return cudaErrorInvalidValue;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.units = units_of(docs, Lo, ws);
  a.H = pr.H;
  a.hq_div = (int32_t)(pr.H / pr.Hqk);
  a.gate_head = pr.gate_head;
  a.vd = (int32_t)pr.V;
  a.scale = pr.scale;
  a.g = pr.g;
  a.h0 = pr.h0;
  a.ht = ht;
  a.o = (__nv_bfloat16 *)o;
  a.err = pr.err;
  const int smem = fsm::BYTES + 1024;
  cudaError_t e;
  auto *kernel = a.gate_head ? gla_fwd_kernel<true> : gla_fwd_kernel<false>;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  const dim3 grid((unsigned)(2 * Lo.max_units * pr.H));
  if (Lo.pieces && Lo.table &&
      (e = launch_build_units(docs, Lo.plen, (Unit *)(ws + Lo.off_units), Lo.max_units, st)) != cudaSuccess)
    return e;
  if (a.units.order &&
      (e = launch_order_units(a.units, Lo.max_units, (int32_t *)(ws + Lo.off_order), st)) != cudaSuccess)
    return e;
  if (Lo.pieces) {
    a.lbuf = (float *)(ws + Lo.off_L);
    a.dbuf = (float *)(ws + Lo.off_D);
    FwdArgs as = a;
    as.ht = nullptr;
    if ((e = launch_piece_states(maps, as, nullptr, nullptr, Lo.max_units, pr.H, st)) != cudaSuccess) return e;
  }
  if ((e = launch_pairs(kernel, grid, smem, st, maps, a)) != cudaSuccess) return e;
  mark_launch("gla_fwd_kernel", st);
  return cudaSuccess;
}

cudaError_t doc_states(const Prob &pr, const Docs &docs, const void *dO, float *L, float *D, cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
  if (const cudaError_t be = bind_context()) return be;
  const int64_t BT = pr.BT;
  FwdMaps fm, rm;
  memset(&fm, 0, sizeof(fm));
  if (!make_map(&fm.q, pr.q, true, KD, pr.Hqk, BT, 64, pr.qs) ||
      !make_map(&fm.k, pr.k, true, KD, pr.Hqk, BT, 64, pr.ks) ||
      !make_map(&fm.v, pr.v, true, pr.V, pr.H, BT, 64, pr.vs) ||
      (!pr.gate_head && !make_map(&fm.g, pr.g, false, KD, pr.H, BT, 32)))
    return cudaErrorInvalidValue;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.units.docs = docs;  // one unit per document, index order
  a.H = pr.H;
  a.hq_div = (int32_t)(pr.H / pr.Hqk);
  a.gate_head = pr.gate_head;
  a.vd = (int32_t)pr.V;
  a.scale = pr.scale;
  a.g = pr.g;
  a.err = pr.err;
  a.lbuf = L;
  a.dbuf = D;
  a.all_units = 1;
  cudaError_t e;
  if (!dO) {
    e = launch_piece_states(fm, a, nullptr, nullptr, docs.n, pr.H, st);
  } else {
    rm = fm;
    rm.k = fm.q;  // the reverse pass runs q through the k slot and do through the v slot
    if (!make_map(&rm.v, dO, true, pr.V, pr.H, BT, 64)) return cudaErrorInvalidValue;
    e = launch_piece_states(rm, a, &rm, &a, docs.n, pr.H, st, true);
  }
  return e;
}

}  // namespace tc
}  // namespace glacore
