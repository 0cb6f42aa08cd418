// internal.cuh -- declarations shared by the host library and its kernels.
// Nothing here is part of the public ABI (include/glacore.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/glacore.h"

namespace glacore {

// Device error word: the first device-detected error code (glacore_status)
// is kept until glacore_get_device_error reads and clears it.  Kernels get
// its address as an argument (the word itself lives in api.cu).
__device__ __forceinline__ void set_device_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Document table.  Without segment_ids every batch row is one document
// (start = d * T).  With segment_ids the prep kernel fills `start`
// ([n+1] flattened token offsets) and `cbase` ([n+1] first chunk slot of
// each document for the state workspace, for chunk length `chunk`).
struct Docs {
  const int64_t *start;  // nullptr: rows
  const int64_t *cbase;  // nullptr: rows
  int64_t T;             // row length
  int64_t n;             // number of documents (grid size)
  int chunk;             // chunk length the cbase table was built for

  __device__ __forceinline__ void range(int64_t d, int64_t &s, int64_t &e) const {
    if (start) {
      s = start[d];
      e = start[d + 1];
    } else {
      s = d * T;
      e = s + T;
    }
  }
  __device__ __forceinline__ int64_t chunk_base(int64_t d) const {
    return cbase ? cbase[d] : d * ((T + chunk - 1) / chunk);
  }
};

// A unit of work of the tensor-core kernels: tokens [start, end) of one
// document, the `piece`-th of the `npieces` consecutive pieces the document
// is split into (exact sequence split: the state entering a piece comes from
// a scan over the pieces' local end states).
struct Unit {
  int64_t start, end;
  int32_t doc, piece, npieces, pad;
};

// Units of a launch: an explicit table (pieces of packed documents); with
// `table` null and plen > 0, rows of docs.T tokens each cut into pieces of
// plen tokens (unit u = piece u % n of row u / n); otherwise one unit per
// document of `docs`.
struct Units {
  const Unit *table;
  Docs docs;
  int64_t plen;
  const int32_t *order;  // launch order (longest first) or null (unit index order)
  __device__ __forceinline__ int64_t at(int64_t r) const { return order ? (int64_t)order[r] : r; }
  __device__ __forceinline__ Unit get(int64_t u) const {
    if (table) return table[u];
    Unit r;
    r.pad = 0;
    if (plen > 0) {
      const int64_t np = (docs.T + plen - 1) / plen, d = u / np, p = u - d * np;
      r.start = d * docs.T + p * plen;
      r.end = min(r.start + plen, (d + 1) * docs.T);
      r.doc = (int32_t)d;
      r.piece = (int32_t)p;
      r.npieces = (int32_t)np;
      return r;
    }
    docs.range(u, r.start, r.end);
    r.doc = (int32_t)u;
    r.piece = 0;
    r.npieces = 1;
    return r;
  }
};

// Exclusive block-wide prefix sum (all threads of the block call it; warp
// sums in `warp_buf[32]`); `total` receives the block total.
__device__ __forceinline__ int64_t block_excl_scan(int64_t x, int64_t *warp_buf, int64_t &total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int64_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_buf[w] = inc;
  __syncthreads();
  if (w == 0) {
    int64_t s = lane < nw ? warp_buf[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nw) warp_buf[lane] = s;  // inclusive warp prefix
  }
  __syncthreads();
  const int64_t before = w ? warp_buf[w - 1] : 0;
  total = warp_buf[nw - 1];
  __syncthreads();
  return before + inc - x;
}

// Problem as the kernels see it (token axis flattened: BT = B * T).
struct Prob {
  int64_t BT, H, Hqk, K, V;
  int64_t qs, ks, vs;  // elements between consecutive tokens of q, k, v
  int gate_head;  // 0: g[BT,H,K]; 1: g[BT,H]
  float scale;
  const void *q, *k, *v;
  const float *g;
  const float *h0;
  int *err;  // device error word
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---- SIMT path (fp32 arithmetic; chunk of 16, 32 or 64 tokens) ---------
namespace simt {
constexpr int SC_DEFAULT = 16;  // chunk length of the SIMT kernels unless the caller asks for another
constexpr int SV = 32;          // value columns per forward CTA
constexpr size_t kMaxSmem = 227 * 1024;  // dynamic shared memory per CTA

// Forward / state pass with chunks of sc (16, 32 or 64) tokens.  o may be null
// (state pass).  ws_states: if non-null, the fp32 state entering every chunk
// is written to ws_states[(cbase + j) * H + h][K][V].  ht: final state or null.
cudaError_t launch_fwd(const Prob &p, const Docs &docs, int dtype, int sc, void *o, float *ht,
                       float *ws_states, cudaStream_t st);
// Backward gradient pass over chunks in reverse (reads ws_states and the
// final states written by the state pass).
cudaError_t launch_bwd(const Prob &p, const Docs &docs, int dtype, int sc, const void *dO,
                       const float *dht, const float *ws_states, const float *ws_final,
                       void *dq, void *dk, float *dq_acc, float *dk_acc, void *dv, float *dg,
                       float *dh0, cudaStream_t st);
cudaError_t launch_convert(const float *src, void *dst, int dtype, int64_t n, cudaStream_t st);
size_t fwd_smem(int64_t K, int sc);
size_t bwd_smem(int64_t K, int64_t V, int sc);
// True when both kernels' shared memory fits for chunks of sc tokens.
bool chunk_fits(int64_t K, int64_t V, int sc);
}  // namespace simt

// SSD through the GLA tensor-core kernels (ssd_gla.cu): the states padded
// to V = 128 and back, the per-head dq / dk summed over each q / k group,
// dg summed over K.
namespace ssdx {
cudaError_t pad_states(int64_t mats, int64_t V, const float *src, float *dst, cudaStream_t st);
cudaError_t cut_states(int64_t mats, int64_t V, const float *src, float *dst, cudaStream_t st);
cudaError_t reduce_heads(int64_t BT, int64_t H, int64_t Hqk, const void *x, void *out, cudaStream_t st);
cudaError_t sum_channels(int64_t rows, const float *x, float *dg, cudaStream_t st);
}  // namespace ssdx

// Records the next caller-provided timing event (if any) after a launch.
void mark_launch(const char *label, cudaStream_t st);
// Maps a CUDA result to a status, remembering the CUDA error of this host
// thread's last failing call (glacore_last_cuda_error).
glacore_status status_of(cudaError_t e);

// ---- segment prep ------------------------------------------------------
cudaError_t launch_prep(const int32_t *seg, int64_t B, int64_t T, int64_t n_seqs, int chunk,
                        int64_t *start, int64_t *cbase, int *err, cudaStream_t st);

}  // namespace glacore
