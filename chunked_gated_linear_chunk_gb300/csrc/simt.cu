// simt.cu -- fp32-arithmetic (CUDA-core) chunk kernels.
//
// This is the instance used for fp32 inputs (where tensor-core bf16/tf32
// rounding would exceed a 1e-4 relative error) and for head sizes the
// tensor-core kernels do not cover, and for any problem whose caller asks
// for chunk_size 16 or 32.  It evaluates the same chunk formulas as the
// tensor-core path with chunks of SC = 16, 32 or 64 tokens (a template
// parameter; 16 unless the caller asks otherwise): the short chunk keeps
// the per-chunk decay factors inside the fp32 exponent range for much
// stronger decay.  A chunk whose summed log-decay in some channel is below
// -80 sets GLACORE_ERR_RANGE (exp(-G) would approach the fp32 limit of
// about exp(88)).
//
//   FLAT blog, "Linear Attention / Forward Recurrence" (chunkwise form) and
//   "Gated Linear Attention" (decay ratios as exponentiated chunk-local
//   prefix sums of the log gate):
//     G  = inclusive prefix sum of g inside the chunk, Gam = G at its end
//     qt = scale q exp(G),  kt = k exp(-G),  P = (qt kt^T) masked to s <= t
//     O  = qt S + P V,      S <- diag(exp(Gam)) (S + kt^T V)
//   FLAT blog, "Backward Recurrence" / "Backward Kernels" (reverse chunk
//   walk carrying the state gradient, gate gradient as a suffix sum):
//     dP = (dO V^T) masked, dHh = diag(exp(Gam)) dH
//     dq = scale exp(G) (dO S^T + dP kt),  dk = exp(-G) (dP^T qt + V dHh^T)
//     dv = P^T dO + kt dHh,                 dH <- dHh + qt^T dO
//     dg_t = sum over the rest of the document of (q dq - k dk) plus
//            (S_T (.) dht) 1_V.
#include <algorithm>

#include "internal.cuh"

namespace glacore {
namespace simt {

template <typename T>
__device__ __forceinline__ float ld(const void *p, int64_t i) {
  return to_f32(reinterpret_cast<const T *>(p)[i]);
}

__device__ __forceinline__ float gate_at(const Prob &p, int64_t tok, int64_t h, int64_t c) {
  return p.gate_head ? p.g[tok * p.H + h] : p.g[(tok * p.H + h) * p.K + c];
}

size_t fwd_smem(int64_t K, int SC) {
  return sizeof(float) * (size_t)(K * SV + 2 * SC * K + SC * SV + SC * SC + K);
}

// Lowest summed log-decay of one chunk in one channel that the chunk
// formulas keep inside the fp32 exponent range.
constexpr float kMinChunkLogDecay = -80.f;

// grid (n_docs, H, ceil(V / SV)), 256 threads.
template <typename T, int SC>
__global__ void __launch_bounds__(256) fwd_kernel(Prob p, Docs docs, T *o, float *ht, float *ws) {
  const int64_t d = blockIdx.x, h = blockIdx.y, v0 = (int64_t)blockIdx.z * SV;
  const int64_t K = p.K, V = p.V;
  const int nv = (int)min((int64_t)SV, V - v0);
  const int64_t hk = h / (p.H / p.Hqk);
  int64_t s0, s1;
  docs.range(d, s0, s1);
  const int64_t cb = docs.chunk_base(d);
  extern __shared__ float sm[];
  float *S = sm;             // [K][SV]
  float *qt = S + K * SV;    // [SC][K]
  float *kt = qt + SC * K;   // [SC][K]
  float *vt = kt + SC * K;   // [SC][SV]
  float *P = vt + SC * SV;   // [SC][SC]
  float *gam = P + SC * SC;  // [K]
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int64_t i = tid; i < K * SV; i += nt) {
    const int64_t c = i / SV;
    const int j = (int)(i % SV);
    S[i] = (p.h0 && j < nv) ? p.h0[((d * p.H + h) * K + c) * V + v0 + j] : 0.f;
  }
  __syncthreads();
  int64_t jc = 0;
  for (int64_t a0 = s0; a0 < s1; a0 += SC, ++jc) {
    const int L = (int)min((int64_t)SC, s1 - a0);
    if (ws) {
      float *dst = ws + ((cb + jc) * p.H + h) * K * V;
      for (int64_t i = tid; i < K * nv; i += nt) {
        const int64_t c = i / nv;
        const int j = (int)(i % nv);
        dst[c * V + v0 + j] = S[c * SV + j];
      }
    }
    for (int64_t c = tid; c < K; c += nt) {
      float G = 0.f;
      for (int t = 0; t < SC; ++t) {
        if (t < L) {
          const int64_t tok = a0 + t;
          G += gate_at(p, tok, h, c);
          const int64_t qo = hk * K + c;
          qt[t * K + c] = p.scale * ld<T>(p.q, tok * p.qs + qo) * expf(G);
          kt[t * K + c] = ld<T>(p.k, tok * p.ks + qo) * expf(-G);
        } else {
          qt[t * K + c] = 0.f;
          kt[t * K + c] = 0.f;
        }
      }
      gam[c] = G;
      if (!(G >= kMinChunkLogDecay)) set_device_error(p.err, GLACORE_ERR_RANGE);
    }
    for (int i = tid; i < SC * SV; i += nt) {
      const int t = i / SV, j = i % SV;
      vt[i] = (t < L && j < nv) ? ld<T>(p.v, (a0 + t) * p.vs + h * V + v0 + j) : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < SC * SC; i += nt) {
      const int t = i / SC, s = i % SC;
      float acc = 0.f;
      if (s <= t && t < L)
        for (int64_t c = 0; c < K; ++c) acc += qt[t * K + c] * kt[s * K + c];
      P[i] = acc;
    }
    __syncthreads();
    if (o) {
      for (int i = tid; i < SC * SV; i += nt) {
        const int t = i / SV, j = i % SV;
        if (t < L && j < nv) {
          float acc = 0.f;
          for (int64_t c = 0; c < K; ++c) acc += qt[t * K + c] * S[c * SV + j];
          for (int s = 0; s <= t; ++s) acc += P[t * SC + s] * vt[s * SV + j];
          o[((a0 + t) * p.H + h) * V + v0 + j] = from_f32<T>(acc);
        }
      }
    }
    __syncthreads();
    for (int64_t i = tid; i < K * SV; i += nt) {
      const int64_t c = i / SV;
      const int j = (int)(i % SV);
      float acc = S[i];
      for (int s = 0; s < L; ++s) acc += kt[s * K + c] * vt[s * SV + j];
      S[i] = expf(gam[c]) * acc;
    }
    __syncthreads();
  }
  if (ht) {
    for (int64_t i = tid; i < K * nv; i += nt) {
      const int64_t c = i / nv;
      const int j = (int)(i % nv);
      ht[((d * p.H + h) * K + c) * V + v0 + j] = S[c * SV + j];
    }
  }
}

size_t bwd_smem(int64_t K, int64_t V, int SC) {
  return sizeof(float) * (size_t)(2 * K * V + 8 * SC * K + 2 * SC * V + 2 * SC * SC + 2 * K + SC);
}

// grid (n_docs, H), 256 threads.  Reads the fp32 chunk-entry states
// (ws) and the final states (wsfin) written by the state pass.
template <typename T, int SC>
__global__ void __launch_bounds__(256)
    bwd_kernel(Prob p, Docs docs, const T *dO, const float *dht, const float *ws,
               const float *wsfin, T *dq, T *dk, float *dq_acc, float *dk_acc, T *dv, float *dg,
               float *dh0) {
  const int64_t d = blockIdx.x, h = blockIdx.y;
  const int64_t K = p.K, V = p.V, H = p.H;
  const int64_t hk = h / (H / p.Hqk);
  int64_t s0, s1;
  docs.range(d, s0, s1);
  const int64_t cb = docs.chunk_base(d);
  extern __shared__ float sm[];
  float *dH = sm;               // [K][V]
  float *Sp = dH + K * V;       // [K][V]
  float *q_ = Sp + K * V;       // [SC][K] raw q
  float *k_ = q_ + SC * K;      // [SC][K] raw k
  float *qt = k_ + SC * K;      // [SC][K]
  float *kt = qt + SC * K;      // [SC][K]
  float *eG = kt + SC * K;      // [SC][K] exp(G)
  float *eGi = eG + SC * K;     // [SC][K] exp(-G)
  float *dqs = eGi + SC * K;    // [SC][K]
  float *dks = dqs + SC * K;    // [SC][K]
  float *vv = dks + SC * K;     // [SC][V]
  float *dd = vv + SC * V;      // [SC][V]
  float *P = dd + SC * V;       // [SC][SC]
  float *dP = P + SC * SC;      // [SC][SC]
  float *carry = dP + SC * SC;  // [K]
  float *gam = carry + K;       // [K]
  float *dgt = gam + K;         // [SC]
  const int tid = threadIdx.x, nt = blockDim.x;
  const float *dht_dh = dht ? dht + (d * H + h) * K * V : nullptr;
  const float *fin = wsfin + (d * H + h) * K * V;
  for (int64_t i = tid; i < K * V; i += nt) dH[i] = dht_dh ? dht_dh[i] : 0.f;
  for (int64_t c = tid; c < K; c += nt) {
    float acc = 0.f;
    if (dht_dh)
      for (int64_t e = 0; e < V; ++e) acc += fin[c * V + e] * dht_dh[c * V + e];
    carry[c] = acc;  // (S_T (.) dht) 1_V
  }
  const int64_t nch = (s1 - s0 + SC - 1) / SC;
  for (int64_t jc = nch - 1; jc >= 0; --jc) {
    const int64_t a0 = s0 + jc * SC;
    const int L = (int)min((int64_t)SC, s1 - a0);
    const float *src = ws + ((cb + jc) * H + h) * K * V;
    for (int64_t i = tid; i < K * V; i += nt) Sp[i] = src[i];
    for (int64_t c = tid; c < K; c += nt) {
      float G = 0.f;
      for (int t = 0; t < SC; ++t) {
        const int64_t idx = t * K + c;
        if (t < L) {
          const int64_t tok = a0 + t;
          G += gate_at(p, tok, h, c);
          const int64_t qo = hk * K + c;
          const float qv = ld<T>(p.q, tok * p.qs + qo), kv = ld<T>(p.k, tok * p.ks + qo);
          const float e = expf(G), ei = expf(-G);
          q_[idx] = qv;
          k_[idx] = kv;
          eG[idx] = e;
          eGi[idx] = ei;
          qt[idx] = p.scale * qv * e;
          kt[idx] = kv * ei;
        } else {
          q_[idx] = k_[idx] = qt[idx] = kt[idx] = eG[idx] = eGi[idx] = 0.f;
        }
      }
      gam[c] = G;
      if (!(G >= kMinChunkLogDecay)) set_device_error(p.err, GLACORE_ERR_RANGE);
    }
    for (int64_t i = tid; i < SC * V; i += nt) {
      const int t = (int)(i / V);
      const int64_t e = i % V;
      const int64_t off = ((a0 + t) * H + h) * V + e;
      vv[i] = t < L ? ld<T>(p.v, (a0 + t) * p.vs + h * V + e) : 0.f;
      dd[i] = t < L ? to_f32(dO[off]) : 0.f;
    }
    if (tid < SC) dgt[tid] = 0.f;
    __syncthreads();
    for (int i = tid; i < SC * SC; i += nt) {
      const int t = i / SC, s = i % SC;
      float a = 0.f, b = 0.f;
      if (s <= t && t < L) {
        for (int64_t c = 0; c < K; ++c) a += qt[t * K + c] * kt[s * K + c];
        for (int64_t e = 0; e < V; ++e) b += dd[t * V + e] * vv[s * V + e];
      }
      P[i] = a;
      dP[i] = b;
    }
    for (int64_t i = tid; i < K * V; i += nt) dH[i] *= expf(gam[i / V]);  // dHh
    __syncthreads();
    for (int64_t i = tid; i < SC * K; i += nt) {
      const int t = (int)(i / K);
      const int64_t c = i % K;
      float a = 0.f, b = 0.f;
      if (t < L) {
        for (int64_t e = 0; e < V; ++e) a += dd[t * V + e] * Sp[c * V + e];
        for (int s = 0; s <= t; ++s) a += dP[t * SC + s] * kt[s * K + c];
        // dk at position t (as the key index s = t)
        for (int u = t; u < L; ++u) b += dP[u * SC + t] * qt[u * K + c];
        for (int64_t e = 0; e < V; ++e) b += vv[t * V + e] * dH[c * V + e];
      }
      dqs[i] = p.scale * eG[i] * a;
      dks[i] = eGi[i] * b;
    }
    for (int64_t i = tid; i < SC * V; i += nt) {
      const int s = (int)(i / V);
      const int64_t e = i % V;
      if (s < L) {
        float a = 0.f;
        for (int t = s; t < L; ++t) a += P[t * SC + s] * dd[t * V + e];
        for (int64_t c = 0; c < K; ++c) a += kt[s * K + c] * dH[c * V + e];
        dv[((a0 + s) * H + h) * V + e] = from_f32<T>(a);
      }
    }
    __syncthreads();
    for (int64_t c = tid; c < K; c += nt) {
      float acc = carry[c];
      for (int t = L - 1; t >= 0; --t) {
        const int64_t idx = t * K + c;
        acc += q_[idx] * dqs[idx] - k_[idx] * dks[idx];
        if (p.gate_head)
          atomicAdd(&dgt[t], acc);
        else
          dg[((a0 + t) * H + h) * K + c] = acc;
      }
      carry[c] = acc;
    }
    for (int64_t i = tid; i < SC * K; i += nt) {
      const int t = (int)(i / K);
      const int64_t c = i % K;
      if (t < L) {
        const int64_t qi = ((a0 + t) * p.Hqk + hk) * K + c;
        if (dq_acc) {
          atomicAdd(&dq_acc[qi], dqs[i]);
          atomicAdd(&dk_acc[qi], dks[i]);
        } else {
          dq[qi] = from_f32<T>(dqs[i]);
          dk[qi] = from_f32<T>(dks[i]);
        }
      }
    }
    for (int64_t i = tid; i < K * V; i += nt) {
      const int64_t c = i / V, e = i % V;
      float a = dH[i];
      for (int t = 0; t < L; ++t) a += qt[t * K + c] * dd[t * V + e];
      dH[i] = a;
    }
    __syncthreads();
    if (p.gate_head && tid < L) dg[(a0 + tid) * H + h] = dgt[tid];
    __syncthreads();
  }
  if (dh0)
    for (int64_t i = tid; i < K * V; i += nt) dh0[(d * H + h) * K * V + i] = dH[i];
}

template <typename T>
__global__ void convert_kernel(const float *src, T *dst, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = from_f32<T>(src[i]);
}

template <typename T, int SC>
static cudaError_t fwd_as(const Prob &p, const Docs &docs, void *o, float *ht, float *ws_states,
                          cudaStream_t st) {
  dim3 grid((unsigned)docs.n, (unsigned)p.H, (unsigned)((p.V + SV - 1) / SV));
  const size_t smem = fwd_smem(p.K, SC);
  auto k = fwd_kernel<T, SC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<grid, 256, smem, st>>>(p, docs, (T *)o, ht, ws_states);
  mark_launch(o ? "simt_fwd" : "simt_state_pass", st);
  return cudaGetLastError();
}

bool chunk_fits(int64_t K, int64_t V, int sc) {
  return (sc == 16 || sc == 32 || sc == 64) && fwd_smem(K, sc) <= kMaxSmem && bwd_smem(K, V, sc) <= kMaxSmem;
}

cudaError_t launch_fwd(const Prob &p, const Docs &docs, int dtype, int sc, void *o, float *ht,
                       float *ws_states, cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
  if (dtype == GLACORE_BF16) {
    using T = __nv_bfloat16;
    return sc == 64   ? fwd_as<T, 64>(p, docs, o, ht, ws_states, st)
           : sc == 32 ? fwd_as<T, 32>(p, docs, o, ht, ws_states, st)
                      : fwd_as<T, 16>(p, docs, o, ht, ws_states, st);
  }
  using T = float;
  return sc == 64   ? fwd_as<T, 64>(p, docs, o, ht, ws_states, st)
         : sc == 32 ? fwd_as<T, 32>(p, docs, o, ht, ws_states, st)
                    : fwd_as<T, 16>(p, docs, o, ht, ws_states, st);
}

template <typename T, int SC>
static cudaError_t bwd_as(const Prob &p, const Docs &docs, const void *dO, const float *dht,
                          const float *ws_states, const float *ws_final, void *dq, void *dk,
                          float *dq_acc, float *dk_acc, void *dv, float *dg, float *dh0, cudaStream_t st) {
  dim3 grid((unsigned)docs.n, (unsigned)p.H);
  const size_t smem = bwd_smem(p.K, p.V, SC);
  auto k = bwd_kernel<T, SC>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<grid, 256, smem, st>>>(p, docs, (const T *)dO, dht, ws_states, ws_final, (T *)dq, (T *)dk, dq_acc,
                             dk_acc, (T *)dv, dg, dh0);
  mark_launch("simt_bwd", st);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const Prob &p, const Docs &docs, int dtype, int sc, const void *dO,
                       const float *dht, const float *ws_states, const float *ws_final, void *dq,
                       void *dk, float *dq_acc, float *dk_acc, void *dv, float *dg, float *dh0,
                       cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
#define GLACORE_SIMT_BWD(T, SCV) \
  bwd_as<T, SCV>(p, docs, dO, dht, ws_states, ws_final, dq, dk, dq_acc, dk_acc, dv, dg, dh0, st)
  if (dtype == GLACORE_BF16) {
    using T = __nv_bfloat16;
    return sc == 64 ? GLACORE_SIMT_BWD(T, 64) : sc == 32 ? GLACORE_SIMT_BWD(T, 32) : GLACORE_SIMT_BWD(T, 16);
  }
  using T = float;
  return sc == 64 ? GLACORE_SIMT_BWD(T, 64) : sc == 32 ? GLACORE_SIMT_BWD(T, 32) : GLACORE_SIMT_BWD(T, 16);
#undef GLACORE_SIMT_BWD
}

cudaError_t launch_convert(const float *src, void *dst, int dtype, int64_t n, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int blocks = (int)std::min<int64_t>((n + 255) / 256, 4096);
  if (dtype == GLACORE_BF16)
    convert_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(src, (__nv_bfloat16 *)dst, n);
  else
    convert_kernel<float><<<blocks, 256, 0, st>>>(src, (float *)dst, n);
  mark_launch("convert", st);
  return cudaGetLastError();
}

}  // namespace simt
}  // namespace glacore
