// api.cu -- the C ABI (include/glacore.h): validation, workspace layout,
// segment preparation and kernel launches.  All compute runs in the
// kernels; this file only checks arguments and enqueues work.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "internal.cuh"
#include "tc.cuh"
#include "tc_ssd.cuh"
#include "tc_ptx.cuh"

namespace glacore {

__device__ int g_device_error = 0;

// Optional per-launch timing marks (measurement hook used by the bench):
// after each kernel launch of a call, the next caller-provided event is
// recorded on the call's stream.  Thread-local; off unless set.
static thread_local cudaEvent_t *t_events = nullptr;
static thread_local int t_nev = 0, t_used = 0;
static thread_local const char *t_labels[64];

static thread_local cudaError_t t_last_cuda = cudaSuccess;
glacore_status status_of(cudaError_t e) {
  if (e == cudaSuccess) return GLACORE_OK;
  t_last_cuda = e;
  return GLACORE_ERR_CUDA;
}

void mark_launch(const char *label, cudaStream_t st) {
  if (t_events && t_used < t_nev) {
    cudaEventRecord(t_events[t_used], st);
    if (t_used < 64) t_labels[t_used] = label;
    ++t_used;
  }
}

// Device address of g_device_error for the current device (looked up once
// per device; kernels receive it as an argument).  The cache entries are
// atomics: host threads may look the address up concurrently (they store
// the same value).
static int *device_error_ptr() {
  static std::atomic<int *> cache[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  int *p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    p = (int *)ptr;
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

// ---- segment preparation (one CTA; documents numbered row-major) ------
//
// JLA product page (karlex.ai/jla): segment_ids make a packed batch train
// exactly as its documents one by one.  A document starts at t = 0 of each
// row and wherever the id changes from the previous token of the row.

__global__ void __launch_bounds__(1024) prep_kernel(const int32_t *seg, int64_t B, int64_t T,
                                                    int64_t n_seqs, int chunk, int64_t *start,
                                                    int64_t *cbase, int *err) {
  __shared__ int64_t wbuf[32];
  const int64_t BT = B * T;
  constexpr int TPT = 16;  // consecutive tokens per thread and pass
  int64_t off = 0;
  for (int64_t base = 0; base < BT; base += (int64_t)blockDim.x * TPT) {
    const int64_t p0 = base + (int64_t)threadIdx.x * TPT;
    uint32_t flags = 0;
    int64_t cnt = 0;
    int64_t col = p0 % T;
    int32_t prev = (p0 > 0 && p0 < BT) ? seg[p0 - 1] : 0;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      const int64_t pos = p0 + i;
      if (pos < BT) {
        const int32_t cur = seg[pos];
        const bool f = col == 0 || cur != prev;
        flags |= (uint32_t)f << i;
        cnt += f;
        prev = cur;
      }
      if (++col == T) col = 0;
    }
    int64_t tot;
    int64_t idx = off + block_excl_scan(cnt, wbuf, tot);
#pragma unroll
    for (int i = 0; i < TPT; ++i)
      if ((flags >> i) & 1u) {
        if (idx < n_seqs) start[idx] = p0 + i;
        ++idx;
      }
    off += tot;
  }
  const int64_t count = off;
  if (threadIdx.x == 0 && count != n_seqs) set_device_error(err, GLACORE_ERR_DOCS);
  // documents that segment_ids does not have become empty; the table always
  // ends at BT so that every kernel stays inside the token range
  for (int64_t i = count + threadIdx.x; i < n_seqs; i += blockDim.x) start[i] = BT;
  if (threadIdx.x == 0) start[n_seqs] = BT;
  __syncthreads();
  int64_t coff = 0;
  for (int64_t base = 0; base < n_seqs; base += blockDim.x) {
    const int64_t d = base + threadIdx.x;
    int64_t nch = 0;
    if (d < n_seqs) nch = (start[d + 1] - start[d] + chunk - 1) / chunk;
    int64_t tot;
    const int64_t ex = block_excl_scan(nch, wbuf, tot);
    if (d < n_seqs) cbase[d] = coff + ex;
    coff += tot;
  }
  if (threadIdx.x == 0) cbase[n_seqs] = coff;
}

__global__ void count_kernel(const int32_t *seg, int64_t B, int64_t T, unsigned long long *out) {
  const int64_t BT = B * T;
  unsigned long long local = 0;
  for (int64_t pos = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; pos < BT;
       pos += (int64_t)gridDim.x * blockDim.x)
    local += (pos % T == 0) || (seg[pos] != seg[pos - 1]);
  for (int o = 16; o; o >>= 1) local += __shfl_down_sync(0xffffffffu, local, o);
  if ((threadIdx.x & 31) == 0 && local) atomicAdd(out, local);
}

cudaError_t launch_prep(const int32_t *seg, int64_t B, int64_t T, int64_t n_seqs, int chunk,
                        int64_t *start, int64_t *cbase, int *err, cudaStream_t st) {
  prep_kernel<<<1, 1024, 0, st>>>(seg, B, T, n_seqs, chunk, start, cbase, err);
  mark_launch("segment_prep", st);
  return cudaGetLastError();
}

// ---- self-test of the bounded waits -------------------------------------
//
// One thread waits, through the kernels' own bounded wait (ptx::mbar_wait),
// on a shared-memory mbarrier that nothing ever arrives on: phase 0 never
// completes, the limit runs out and the timeout is recorded exactly as a
// kernel records it.  No copy, MMA or tensor memory is in flight.
__global__ void wait_selftest_kernel(long long cycles, int *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, cycles)) set_device_error(err, GLACORE_ERR_TIMEOUT);
}

// ---- exact hand-off of states between sequence pieces ------------------
//
// JLA product page ("our split is exact"): the recurrence is linear in the
// state, so the state entering piece r is the fold of the earlier pieces'
// local end states L and total decays D, and the state gradient leaving
// piece r the fold of the later pieces' local start-state gradients and
// decays.  One thread per state element, the pieces in order.
__global__ void state_scan_kernel(const float *L, const float *D, int64_t R, int64_t mats, int64_t K, int64_t V,
                                  const float *seed, int64_t r, int reverse, float *out) {
  const int64_t n = mats * K * V;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t mk = i / V;  // (matrix, key row)
    float s = seed ? seed[i] : 0.f;
    if (!reverse) {
      for (int64_t q = 0; q < r; ++q) s = D[q * mats * K + mk] * s + L[q * n + i];
    } else {
      for (int64_t q = R - 1; q > r; --q) s = D[q * mats * K + mk] * s + L[q * n + i];
    }
    out[i] = s;
  }
}

// ---- argument checks ----------------------------------------------------

namespace {

struct Layout {
  bool ssd;            // SSD tensor-core kernels (one gate per head, V = 64)
  bool tc;             // tensor-core path
  bool ssdx;           // SSD through the GLA tensor-core kernels (states padded in the workspace)
  int chunk;           // chunk length of the state workspace / doc table
  size_t off_start, off_cbase;  // doc tables (segments only)
  size_t off_states, off_final, off_acc_q, off_acc_k, off_tc;
  // ssdx: the GLA problem's tensors ([B*T, H, 128]) and states ([n, H, 128, 128])
  size_t off_xh0, off_xht, off_xdht, off_xdq, off_xdk, off_xdg, off_xdh0;
  size_t total;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

glacore_status check_problem(const glacore_problem *p, bool head_gate) {
  if (!p) return GLACORE_ERR_INVALID_ARG;
  if (p->B < 1 || p->T < 0 || p->H < 1 || p->Hqk < 1 || p->K < 1 || p->V < 1)
    return GLACORE_ERR_INVALID_ARG;
  if (p->K > 256 || p->V > 256) return GLACORE_ERR_INVALID_ARG;
  if (p->H % p->Hqk) return GLACORE_ERR_INVALID_ARG;
  if (p->dtype != GLACORE_F32 && p->dtype != GLACORE_BF16) return GLACORE_ERR_INVALID_ARG;
  if (p->reserved0 != 0) return GLACORE_ERR_INVALID_ARG;
  if (p->chunk_size < 0) return GLACORE_ERR_INVALID_ARG;
  if (p->chunk_size != 0 && p->chunk_size != 16 && p->chunk_size != 32 && p->chunk_size != 64)
    return GLACORE_ERR_UNSUPPORTED;
  if (p->B > (int64_t)1 << 31 || p->T > (int64_t)1 << 31 || p->H > 65535)
    return GLACORE_ERR_INVALID_ARG;
  const int64_t BT = p->B * p->T;
  if (!p->segment_ids) {
    if (p->n_seqs != (p->T > 0 ? p->B : 0)) return GLACORE_ERR_INVALID_ARG;
  } else {
    if (p->n_seqs < (BT > 0 ? 1 : 0) || p->n_seqs > BT) return GLACORE_ERR_INVALID_ARG;
  }
  if (BT > 0 && (!p->q || !p->k || !p->v || !p->g)) return GLACORE_ERR_INVALID_ARG;
  if (!(p->scale == p->scale)) return GLACORE_ERR_INVALID_ARG;  // NaN scale
  // token strides of q, k, v: 0 (contiguous) or at least one token's heads
  if (p->q_stride < 0 || p->k_stride < 0 || p->v_stride < 0) return GLACORE_ERR_INVALID_ARG;
  if ((p->q_stride && p->q_stride < p->Hqk * p->K) || (p->k_stride && p->k_stride < p->Hqk * p->K) ||
      (p->v_stride && p->v_stride < p->H * p->V))
    return GLACORE_ERR_INVALID_ARG;
  (void)head_gate;
  return GLACORE_OK;
}

// The CUDA-core kernels take any K, V up to 128 at chunk 16 (chunk_size 0
// or 16), and chunks of 32 or 64 where their shared memory fits.
int simt_chunk(const glacore_problem *p) { return p->chunk_size ? p->chunk_size : simt::SC_DEFAULT; }
bool simt_supported(const glacore_problem *p) {
  return p->K <= 128 && p->V <= 128 && simt::chunk_fits(p->K, p->V, simt_chunk(p));
}

// The shape of the GLA problem an SSD problem is run as (ssd_gla.cu): K and
// V of 128, every head its own q / k.  It is checked and laid out so; the
// kernels then read the grouped q / k, the per-head gate and the V-column v
// and do in place (the columns past V as zeros).
glacore_problem ssd_as_gla(const glacore_problem *p) {
  glacore_problem e = *p;
  e.Hqk = p->H;
  e.K = 128;
  e.V = 128;
  return e;
}
bool ssdx_supported(const glacore_problem *p, bool head_gate, bool backward) {
  // V of 64 or 128: the kernels read v and do as 128 columns, the missing 64
  // zero-filled by TMA, and store o and dv per 64-column half
  if (!head_gate || p->dtype != GLACORE_BF16 || p->K != 128 || (p->V != 64 && p->V != 128)) return false;
  const glacore_problem e = ssd_as_gla(p);
  return tc::supported(&e, false, backward);
}

Layout layout(const glacore_problem *p, bool head_gate, bool backward) {
  Layout L;
  memset(&L, 0, sizeof(L));
  L.ssd = head_gate && ssd::supported(p);
  L.tc = !L.ssd && tc::supported(p, head_gate, backward);
  L.ssdx = !L.ssd && !L.tc && ssdx_supported(p, head_gate, backward);
  L.chunk = (L.ssd || L.tc || L.ssdx) ? tc::C : simt_chunk(p);
  const int64_t BT = p->B * p->T, n = p->n_seqs;
  size_t off = 0;
  if (p->segment_ids) {
    L.off_start = off;
    off = align256(off + sizeof(int64_t) * (n + 1));
    L.off_cbase = off;
    off = align256(off + sizeof(int64_t) * (n + 1));
  }
  if (L.ssd) {
    L.off_tc = off;
    off = align256(off + ssd::workspace_bytes(p, backward));
  } else if (L.ssdx) {
    const size_t rows = (size_t)BT * p->H, bf = rows * 128 * 2, f32 = rows * 128 * 4;
    const size_t st = (size_t)n * p->H * 128 * 128 * 4;
    auto take = [&](size_t &o, size_t bytes) {
      o = off;
      off = align256(off + bytes);
    };
    if (p->initial_state) take(L.off_xh0, st);
    if (!backward) {
      take(L.off_xht, st);
    } else {
      take(L.off_xdht, st);
      take(L.off_xdq, bf);
      take(L.off_xdk, bf);
      take(L.off_xdg, f32);
      if (p->initial_state) take(L.off_xdh0, st);
    }
    const glacore_problem e = ssd_as_gla(p);
    L.off_tc = off;
    off = align256(off + tc::workspace_bytes(&e, false, backward));
  } else if (L.tc) {
    if (backward && p->Hqk != p->H) {
      // shared q / k heads: dq and dk per value head, then summed over the
      // heads of each group
      const size_t bf = (size_t)BT * p->H * 128 * 2;
      L.off_xdq = off;
      off = align256(off + bf);
      L.off_xdk = off;
      off = align256(off + bf);
    }
    L.off_tc = off;
    off = align256(off + tc::workspace_bytes(p, head_gate, backward));
  } else if (backward) {
    const int64_t slots = p->segment_ids ? (BT + L.chunk - 1) / L.chunk + n
                                         : p->B * ((p->T + L.chunk - 1) / L.chunk);
    L.off_states = off;
    off = align256(off + sizeof(float) * (size_t)slots * p->H * p->K * p->V);
    L.off_final = off;
    off = align256(off + sizeof(float) * (size_t)n * p->H * p->K * p->V);
    if (p->Hqk != p->H) {
      L.off_acc_q = off;
      off = align256(off + sizeof(float) * (size_t)BT * p->Hqk * p->K);
      L.off_acc_k = off;
      off = align256(off + sizeof(float) * (size_t)BT * p->Hqk * p->K);
    }
  }
  L.total = off;
  return L;
}

glacore_status check_ws(const glacore_problem *p, const Layout &L) {
  if (L.total == 0) return GLACORE_OK;
  if (!p->workspace || p->workspace_bytes < L.total) return GLACORE_ERR_WORKSPACE;
  if ((uintptr_t)p->workspace & 255) return GLACORE_ERR_WORKSPACE;
  return GLACORE_OK;
}

Prob make_prob(const glacore_problem *p, bool head_gate) {
  Prob q;
  q.BT = p->B * p->T;
  q.H = p->H;
  q.Hqk = p->Hqk;
  q.K = p->K;
  q.V = p->V;
  q.gate_head = head_gate ? 1 : 0;
  q.scale = p->scale;
  q.q = p->q;
  q.k = p->k;
  q.v = p->v;
  q.qs = p->q_stride ? p->q_stride : p->Hqk * p->K;
  q.ks = p->k_stride ? p->k_stride : p->Hqk * p->K;
  q.vs = p->v_stride ? p->v_stride : p->H * p->V;
  q.g = p->g;
  q.h0 = p->initial_state;
  q.err = device_error_ptr();
  return q;
}

glacore_status cuda_status(cudaError_t e) { return status_of(e); }

Docs make_docs(const glacore_problem *p, const Layout &L, char *ws) {
  Docs d;
  d.T = p->T;
  d.n = p->n_seqs;
  d.chunk = L.chunk;
  d.start = p->segment_ids ? (const int64_t *)(ws + L.off_start) : nullptr;
  d.cbase = p->segment_ids ? (const int64_t *)(ws + L.off_cbase) : nullptr;
  return d;
}

glacore_status run_fwd(const glacore_problem *p, bool head_gate, void *o, float *ht,
                       cudaStream_t st) {
  glacore_status s = check_problem(p, head_gate);
  if (s) return s;
  const int64_t BT = p->B * p->T;
  if (BT > 0 && !o) return GLACORE_ERR_INVALID_ARG;
  const Layout L = layout(p, head_gate, false);
  if (!L.ssd && !L.tc && !L.ssdx && !simt_supported(p)) return GLACORE_ERR_UNSUPPORTED;
  if ((s = check_ws(p, L))) return s;
  if ((L.ssd || L.tc || L.ssdx) && !(aligned16(p->q) && aligned16(p->k) && aligned16(p->v) && aligned16(p->g) &&
                aligned16(o) && aligned16(ht) && aligned16(p->initial_state)))
    return GLACORE_ERR_INVALID_ARG;
  if (BT == 0) return GLACORE_OK;
  char *ws = (char *)p->workspace;
  if (p->segment_ids) {
    cudaError_t e = launch_prep(p->segment_ids, p->B, p->T, p->n_seqs, L.chunk,
                                (int64_t *)(ws + L.off_start), (int64_t *)(ws + L.off_cbase),
                                device_error_ptr(), st);
    if (e != cudaSuccess) return status_of(e);
  }
  const Docs docs = make_docs(p, L, ws);
  if (L.ssd) return cuda_status(ssd::fwd(make_prob(p, true), docs, p, o, ht, ws + L.off_tc, st));
  if (L.ssdx) {
    const int64_t mats = p->n_seqs * p->H;
    // q, k of the head groups, the per-head gate and the V-column v are read
    // in place; only the states are padded to V = 128
    glacore_problem e = ssd_as_gla(p);
    e.Hqk = p->Hqk;
    e.V = p->V;
    e.initial_state = p->initial_state ? (const float *)(ws + L.off_xh0) : nullptr;
    cudaError_t c = cudaSuccess;
    if (p->initial_state) c = ssdx::pad_states(mats, p->V, p->initial_state, (float *)(ws + L.off_xh0), st);
    if (c == cudaSuccess)
      c = tc::fwd(make_prob(&e, true), docs, &e, o, ht ? (float *)(ws + L.off_xht) : nullptr, ws + L.off_tc, st);
    if (c == cudaSuccess && ht) c = ssdx::cut_states(mats, p->V, (const float *)(ws + L.off_xht), ht, st);
    return cuda_status(c);
  }
  const Prob pr = make_prob(p, head_gate);
  if (L.tc) return cuda_status(tc::fwd(pr, docs, p, o, ht, ws + L.off_tc, st));
  return cuda_status(simt::launch_fwd(pr, docs, p->dtype, L.chunk, o, ht, nullptr, st));
}

glacore_status run_bwd(const glacore_problem *p, bool head_gate, const void *dO,
                       const float *dht, void *dq, void *dk, void *dv, float *dg, float *dh0,
                       cudaStream_t st) {
  glacore_status s = check_problem(p, head_gate);
  if (s) return s;
  const int64_t BT = p->B * p->T;
  if (BT > 0 && (!dO || !dq || !dk || !dv || !dg)) return GLACORE_ERR_INVALID_ARG;
  const Layout L = layout(p, head_gate, true);
  if (!L.ssd && !L.tc && !L.ssdx && !simt_supported(p)) return GLACORE_ERR_UNSUPPORTED;
  if ((s = check_ws(p, L))) return s;
  if ((L.ssd || L.tc || L.ssdx) && !(aligned16(p->q) && aligned16(p->k) && aligned16(p->v) && aligned16(p->g) &&
                aligned16(dO) && aligned16(dht) && aligned16(dq) && aligned16(dk) &&
                aligned16(dv) && aligned16(dg) && aligned16(dh0) &&
                aligned16(p->initial_state)))
    return GLACORE_ERR_INVALID_ARG;
  if (BT == 0) return GLACORE_OK;
  char *ws = (char *)p->workspace;
  if (p->segment_ids) {
    cudaError_t e = launch_prep(p->segment_ids, p->B, p->T, p->n_seqs, L.chunk,
                                (int64_t *)(ws + L.off_start), (int64_t *)(ws + L.off_cbase),
                                device_error_ptr(), st);
    if (e != cudaSuccess) return status_of(e);
  }
  const Docs docs = make_docs(p, L, ws);
  if (L.ssd)
    return cuda_status(ssd::bwd(make_prob(p, true), docs, p, dO, dht, dq, dk, dv, dg, dh0, ws + L.off_tc, st));
  if (L.ssdx) {
    const int64_t rows = BT * p->H, mats = p->n_seqs * p->H;
    // q, k of the head groups, the per-head gate, the V-column v and do are
    // read in place, dv written in place; only the states are padded to V = 128
    glacore_problem e = ssd_as_gla(p);
    e.Hqk = p->Hqk;
    e.V = p->V;
    e.initial_state = p->initial_state ? (const float *)(ws + L.off_xh0) : nullptr;
    cudaError_t c = cudaSuccess;
    if (p->initial_state)
      c = ssdx::pad_states(mats, p->V, p->initial_state, (float *)(ws + L.off_xh0), st);
    if (c == cudaSuccess && dht) c = ssdx::pad_states(mats, p->V, dht, (float *)(ws + L.off_xdht), st);
    if (c == cudaSuccess)
      c = tc::bwd(make_prob(&e, true), docs, &e, dO, dht ? (const float *)(ws + L.off_xdht) : nullptr,
                  ws + L.off_xdq, ws + L.off_xdk, dv, (float *)(ws + L.off_xdg),
                  dh0 ? (float *)(ws + L.off_xdh0) : nullptr, ws + L.off_tc, st);
    if (c == cudaSuccess) c = ssdx::reduce_heads(BT, p->H, p->Hqk, ws + L.off_xdq, dq, st);
    if (c == cudaSuccess) c = ssdx::reduce_heads(BT, p->H, p->Hqk, ws + L.off_xdk, dk, st);
    if (c == cudaSuccess) c = ssdx::sum_channels(rows, (const float *)(ws + L.off_xdg), dg, st);
    if (c == cudaSuccess && dh0) c = ssdx::cut_states(mats, p->V, (const float *)(ws + L.off_xdh0), dh0, st);
    return cuda_status(c);
  }
  const Prob pr = make_prob(p, head_gate);
  if (L.tc && p->Hqk != p->H) {
    cudaError_t c = tc::bwd(pr, docs, p, dO, dht, ws + L.off_xdq, ws + L.off_xdk, dv, dg, dh0, ws + L.off_tc, st);
    if (c == cudaSuccess) c = ssdx::reduce_heads(BT, p->H, p->Hqk, ws + L.off_xdq, dq, st);
    if (c == cudaSuccess) c = ssdx::reduce_heads(BT, p->H, p->Hqk, ws + L.off_xdk, dk, st);
    return cuda_status(c);
  }
  if (L.tc)
    return cuda_status(tc::bwd(pr, docs, p, dO, dht, dq, dk, dv, dg, dh0, ws + L.off_tc, st));
  float *states = (float *)(ws + L.off_states);
  float *fin = (float *)(ws + L.off_final);
  cudaError_t e = simt::launch_fwd(pr, docs, p->dtype, L.chunk, nullptr, fin, states, st);
  if (e != cudaSuccess) return GLACORE_ERR_CUDA;
  float *accq = nullptr, *acck = nullptr;
  if (p->Hqk != p->H) {
    accq = (float *)(ws + L.off_acc_q);
    acck = (float *)(ws + L.off_acc_k);
    const size_t nb = sizeof(float) * (size_t)BT * p->Hqk * p->K;
    if (cudaMemsetAsync(accq, 0, nb, st) != cudaSuccess) return GLACORE_ERR_CUDA;
    if (cudaMemsetAsync(acck, 0, nb, st) != cudaSuccess) return GLACORE_ERR_CUDA;
  }
  e = simt::launch_bwd(pr, docs, p->dtype, L.chunk, dO, dht, states, fin, dq, dk, accq, acck, dv, dg,
                       dh0, st);
  if (e != cudaSuccess) return GLACORE_ERR_CUDA;
  if (accq) {
    const int64_t n = BT * p->Hqk * p->K;
    if (simt::launch_convert(accq, dq, p->dtype, n, st) != cudaSuccess) return GLACORE_ERR_CUDA;
    if (simt::launch_convert(acck, dk, p->dtype, n, st) != cudaSuccess) return GLACORE_ERR_CUDA;
  }
  return GLACORE_OK;
}

size_t ws_size(const glacore_problem *p, bool head_gate, bool backward) {
  if (check_problem(p, head_gate) != GLACORE_OK) return 0;
  return layout(p, head_gate, backward).total;
}

}  // namespace
}  // namespace glacore

using namespace glacore;

extern "C" {

size_t gla_fwd_workspace_size(const glacore_problem *p) { return ws_size(p, false, false); }
size_t gla_bwd_workspace_size(const glacore_problem *p) { return ws_size(p, false, true); }
size_t ssd_fwd_workspace_size(const glacore_problem *p) { return ws_size(p, true, false); }
size_t ssd_bwd_workspace_size(const glacore_problem *p) { return ws_size(p, true, true); }

glacore_status gla_fwd(const glacore_problem *p, void *o, float *final_state,
                       glacore_stream_t stream) {
  t_used = 0;
  return run_fwd(p, false, o, final_state, (cudaStream_t)stream);
}
glacore_status ssd_fwd(const glacore_problem *p, void *o, float *final_state,
                       glacore_stream_t stream) {
  t_used = 0;
  return run_fwd(p, true, o, final_state, (cudaStream_t)stream);
}
glacore_status gla_bwd(const glacore_problem *p, const void *do_, const float *dht, void *dq,
                       void *dk, void *dv, float *dg, float *dh0, glacore_stream_t stream) {
  t_used = 0;
  return run_bwd(p, false, do_, dht, dq, dk, dv, dg, dh0, (cudaStream_t)stream);
}
glacore_status ssd_bwd(const glacore_problem *p, const void *do_, const float *dht, void *dq,
                       void *dk, void *dv, float *dg, float *dh0, glacore_stream_t stream) {
  t_used = 0;
  return run_bwd(p, true, do_, dht, dq, dk, dv, dg, dh0, (cudaStream_t)stream);
}

glacore_status glacore_count_docs(const int32_t *segment_ids, int64_t B, int64_t T,
                                  int64_t *n_docs, glacore_stream_t stream) {
  if (!n_docs || B < 1 || T < 0 || (B * T > 0 && !segment_ids)) return GLACORE_ERR_INVALID_ARG;
  if (((uintptr_t)n_docs & 7) != 0) return GLACORE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemsetAsync(n_docs, 0, sizeof(int64_t), st) != cudaSuccess) return GLACORE_ERR_CUDA;
  if (B * T == 0) return GLACORE_OK;
  count_kernel<<<256, 256, 0, st>>>(segment_ids, B, T, (unsigned long long *)n_docs);
  return cuda_status(cudaGetLastError());
}

glacore_status glacore_get_device_error(glacore_stream_t stream) {
  cudaStream_t st = (cudaStream_t)stream;
  int h = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&h, g_device_error, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                st) != cudaSuccess)
    return GLACORE_ERR_CUDA;
  if (cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                              st) != cudaSuccess)
    return GLACORE_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GLACORE_ERR_CUDA;
  return (glacore_status)h;
}

glacore_status gla_fwd_state(const glacore_problem *p, float *L, float *D, glacore_stream_t stream) {
  glacore_status s = check_problem(p, false);
  if (s) return s;
  if (p->B * p->T > 0 && (!L || !D)) return GLACORE_ERR_INVALID_ARG;
  if (p->segment_ids || !tc::supported(p, false, false)) return GLACORE_ERR_UNSUPPORTED;
  if (!(aligned16(p->q) && aligned16(p->k) && aligned16(p->v) && aligned16(p->g) && aligned16(L) && aligned16(D)))
    return GLACORE_ERR_INVALID_ARG;
  if (p->B * p->T == 0) return GLACORE_OK;
  t_used = 0;
  Layout Lo;
  memset(&Lo, 0, sizeof(Lo));
  Lo.chunk = tc::C;
  const Docs docs = make_docs(p, Lo, nullptr);
  return cuda_status(tc::doc_states(make_prob(p, false), docs, nullptr, L, D, (cudaStream_t)stream));
}

glacore_status gla_bwd_state(const glacore_problem *p, const void *do_, float *L, float *D,
                             glacore_stream_t stream) {
  glacore_status s = check_problem(p, false);
  if (s) return s;
  if (p->B * p->T > 0 && (!L || !D || !do_)) return GLACORE_ERR_INVALID_ARG;
  if (p->segment_ids || !tc::supported(p, false, true)) return GLACORE_ERR_UNSUPPORTED;
  if (!(aligned16(p->q) && aligned16(p->k) && aligned16(p->v) && aligned16(p->g) && aligned16(L) &&
        aligned16(D) && aligned16(do_)))
    return GLACORE_ERR_INVALID_ARG;
  if (p->B * p->T == 0) return GLACORE_OK;
  t_used = 0;
  Layout Lo;
  memset(&Lo, 0, sizeof(Lo));
  Lo.chunk = tc::C;
  const Docs docs = make_docs(p, Lo, nullptr);
  return cuda_status(tc::doc_states(make_prob(p, false), docs, do_, L, D, (cudaStream_t)stream));
}

glacore_status glacore_state_scan(const float *L, const float *D, int64_t R, int64_t mats, int64_t K, int64_t V,
                                  const float *seed, int64_t r, int32_t reverse, float *out,
                                  glacore_stream_t stream) {
  if (R < 1 || mats < 0 || K < 1 || V < 1 || r < 0 || r >= R || (reverse != 0 && reverse != 1))
    return GLACORE_ERR_INVALID_ARG;
  if (mats == 0) return GLACORE_OK;
  if (!L || !D || !out) return GLACORE_ERR_INVALID_ARG;
  const int64_t n = mats * K * V;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  state_scan_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(L, D, R, mats, K, V, seed, r, reverse, out);
  mark_launch("state_scan", (cudaStream_t)stream);
  return cuda_status(cudaGetLastError());
}

glacore_status glacore_selftest_wait(int64_t cycles, glacore_stream_t stream) {
  if (cycles < 1 || cycles > ((int64_t)1 << 40)) return GLACORE_ERR_INVALID_ARG;
  int *err = device_error_ptr();
  if (!err) return GLACORE_ERR_CUDA;
  wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((long long)cycles, err);
  return cuda_status(cudaGetLastError());
}

const char *glacore_last_cuda_error(void) {
  return t_last_cuda == cudaSuccess ? "no CUDA error" : cudaGetErrorString(t_last_cuda);
}

const char *glacore_status_string(glacore_status s) {
  switch (s) {
    case GLACORE_OK: return "ok";
    case GLACORE_ERR_INVALID_ARG: return "invalid argument";
    case GLACORE_ERR_UNSUPPORTED: return "unsupported configuration";
    case GLACORE_ERR_CUDA: return "CUDA runtime error";
    case GLACORE_ERR_TIMEOUT: return "bounded device wait ran out";
    case GLACORE_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case GLACORE_ERR_DOCS: return "segment_ids holds a different number of documents than n_seqs";
    case GLACORE_ERR_RANGE:
      return "a chunk's summed log-decay is below the kernels' range (-80 per chunk; chunk_size 16 "
             "covers stronger decay)";
  }
  return "unknown status";
}

int glacore_version(void) { return 200; }

void glacore_set_timing_events(void *events, int n_events) {
  t_events = (cudaEvent_t *)events;
  t_nev = events ? n_events : 0;
  t_used = 0;
}
int glacore_timing_count(void) { return t_used; }
const char *glacore_timing_label(int i) {
  return (i >= 0 && i < t_used && i < 64) ? t_labels[i] : "";
}

}  // extern "C"
