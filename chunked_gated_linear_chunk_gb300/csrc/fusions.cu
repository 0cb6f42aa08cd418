// fusions.cu -- the two operations around the recurrence, as fused
// memory-bound kernels with their C ABI (include/glacore.h):
//
// norm_gate: per-head RMSNorm times a swish output gate (FLAT blog,
//   "Full Linear Attention Layer": the layer's output passes a per-head
//   RMSNorm multiplied by a swish output gate, which the page leaves to XLA
//   fusions at 2.3 ms per step).  Over each row of V values:
//       n = o * rsqrt(mean(o^2) + eps),   y = n * w * z * sigmoid(z)
//   backward (r = rsqrt(mean(o^2) + eps), s = sigmoid(z)):
//       dz = dy n w s (1 + z (1 - s)),   dw = sum_rows dy z s n,
//       dn = dy z s w,   do = r dn - r^3 o (dn . o) / V
//
// short_conv: depthwise causal short convolution with bias and SiLU (FLAT
//   blog, "Depthwise Causal Short Convolution"): tap k of Kc reads the input
//   Kc-1-k tokens back, inside the token's document,
//       z_t = b + sum_k W_k x_{t-(Kc-1-k)},   y_t = SiLU(z_t)
//   backward: dz = dy SiLU'(z), SiLU'(z) = s (1 + z (1 - s)); dW_k and db
//   reduce dz times the input the tap reads over every position; dx is the
//   anti-causal correlation of dz with the same taps.
//
// Both are HBM-bound streams: every thread owns 8 consecutive channels (one
// 16-byte vector of bf16) so that a warp reads and writes contiguous rows;
// arithmetic is fp32.  The weight gradients are reduced deterministically:
// per-CTA partial sums in the workspace, then one reduction kernel.
#include <algorithm>

#include "internal.cuh"

namespace glacore {
namespace fuse {

// ---- 8-element vector loads / stores (bf16: 16 bytes, fp32: 32 bytes) ----
__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void ld8(const float *p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4 *>(p)), b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ uint32_t pk(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ void st8(__nv_bfloat16 *p, const float (&v)[8]) {
  *reinterpret_cast<uint4 *>(p) = make_uint4(pk(v[0], v[1]), pk(v[2], v[3]), pk(v[4], v[5]), pk(v[6], v[7]));
}
__device__ __forceinline__ void st8(float *p, const float (&v)[8]) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
// sigmoid with the fast reciprocal-based divide (a few ulp; the outputs are
// rounded to bf16 or checked at 1e-4 in fp32)
__device__ __forceinline__ float sigm(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// ============================================================ norm_gate ====
// A warp step covers 32 / lpr rows (lpr = V / 8 lanes per row); a lane owns
// channels 8 sub .. 8 sub + 7 of its row, so its slice of w stays in
// registers.  Two row steps per iteration keep four 16-byte loads in flight.
constexpr int NG_THREADS = 256;
constexpr int NG_MAX_BLOCKS = 1024;

inline int64_t ng_blocks(int64_t rows, int64_t V) {
  const int64_t rows_per_block = (NG_THREADS / 32) * (32 / (V / 8)) * 2;
  return std::max<int64_t>(1, std::min<int64_t>((rows + rows_per_block - 1) / rows_per_block, NG_MAX_BLOCKS));
}

template <typename T>
__global__ void __launch_bounds__(NG_THREADS)
    norm_gate_fwd_kernel(const T *__restrict__ o, const T *__restrict__ z, const float *__restrict__ w,
                         T *__restrict__ y, int64_t rows, int V, int lg, float eps) {
  const int lane = threadIdx.x & 31, lpr = 1 << lg, sub = lane & (lpr - 1), rpw = 32 >> lg;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float wv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) wv[i] = w[8 * sub + i];
  const float inv_v = 1.f / (float)V;
  for (int64_t r0 = gw * rpw * 2; r0 < rows; r0 += nw * rpw * 2) {
    int64_t row[2];
    float ov[2][8], zv[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      row[u] = r0 + u * rpw + (lane >> lg);
      if (row[u] < rows) {
        ld8(o + row[u] * V + 8 * sub, ov[u]);
        ld8(z + row[u] * V + 8 * sub, zv[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) ov[u][i] = zv[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += ov[u][i] * ov[u][i];
      for (int m = 1; m < lpr; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      const float r = rsqrtf(ss * inv_v + eps);
      float yv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) yv[i] = ov[u][i] * r * wv[i] * zv[u][i] * sigm(zv[u][i]);
      if (row[u] < rows) st8(y + row[u] * V + 8 * sub, yv);
    }
  }
}

// Backward; each CTA writes its partial dw ([V] fp32) to part[blockIdx.x].
template <typename T>
__global__ void __launch_bounds__(NG_THREADS)
    norm_gate_bwd_kernel(const T *__restrict__ o, const T *__restrict__ z, const float *__restrict__ w,
                         const T *__restrict__ dy, T *__restrict__ dox, T *__restrict__ dzx, float *__restrict__ part,
                         int64_t rows, int V, int lg, float eps) {
  __shared__ float red[NG_THREADS / 32][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, lpr = 1 << lg, sub = lane & (lpr - 1),
            rpw = 32 >> lg;
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float wv[8], dwa[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    wv[i] = w[8 * sub + i];
    dwa[i] = 0.f;
  }
  const float inv_v = 1.f / (float)V;
  for (int64_t r0 = gw * rpw * 2; r0 < rows; r0 += nw * rpw * 2) {
    int64_t row[2];
    float ov[2][8], zv[2][8], gv[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      row[u] = r0 + u * rpw + (lane >> lg);
      if (row[u] < rows) {
        ld8(o + row[u] * V + 8 * sub, ov[u]);
        ld8(z + row[u] * V + 8 * sub, zv[u]);
        ld8(dy + row[u] * V + 8 * sub, gv[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) ov[u][i] = zv[u][i] = gv[u][i] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += ov[u][i] * ov[u][i];
      for (int m = 1; m < lpr; m <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
      const float r = rsqrtf(ss * inv_v + eps);
      float dn[8], dzv[8], dot = 0.f;
      const bool live = row[u] < rows;  // padding rows add nothing to dw
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float n = ov[u][i] * r, s = sigm(zv[u][i]), g = zv[u][i] * s;
        const float du = gv[u][i] * g;
        if (live) dwa[i] += du * n;
        dn[i] = du * wv[i];
        dzv[i] = gv[u][i] * n * wv[i] * s * (1.f + zv[u][i] * (1.f - s));
        dot += dn[i] * ov[u][i];
      }
      for (int m = 1; m < lpr; m <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, m);
      const float c = r * r * r * dot * inv_v;
      float dov[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) dov[i] = r * dn[i] - c * ov[u][i];
      if (row[u] < rows) {
        st8(dox + row[u] * V + 8 * sub, dov);
        st8(dzx + row[u] * V + 8 * sub, dzv);
      }
    }
  }
  // dw: lanes of one channel block within the warp, then the warps of the CTA
#pragma unroll
  for (int i = 0; i < 8; ++i)
    for (int m = lpr; m < 32; m <<= 1) dwa[i] += __shfl_xor_sync(0xffffffffu, dwa[i], m);
  if (lane < lpr)
#pragma unroll
    for (int i = 0; i < 8; ++i) red[warp][8 * lane + i] = dwa[i];
  __syncthreads();
  for (int c = threadIdx.x; c < V; c += blockDim.x) {
    float acc = 0.f;
    for (int k = 0; k < NG_THREADS / 32; ++k) acc += red[k][c];
    part[(int64_t)blockIdx.x * V + c] = acc;
  }
}

// out[c] = sum over n partial rows of part[p * stride + c]: block (32, 32),
// x = one of 32 consecutive columns, y = the row phase; each thread adds
// rows y, y + 32, ... in order, then column sums of the 32 phases in phase
// order (deterministic).
__global__ void __launch_bounds__(1024)
    reduce_rows_kernel(const float *__restrict__ part, int64_t n, int64_t stride, int64_t cols, float *__restrict__ out) {
  __shared__ float red[32][33];
  const int64_t c = (int64_t)blockIdx.x * 32 + threadIdx.x;
  float acc = 0.f;
  if (c < cols) {
    int64_t p = threadIdx.y;
    for (; p + 96 < n; p += 128)
      acc += (part[p * stride + c] + part[(p + 32) * stride + c]) +
             (part[(p + 64) * stride + c] + part[(p + 96) * stride + c]);
    for (; p < n; p += 32) acc += part[p * stride + c];
  }
  red[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0 && c < cols) {
    float s2 = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) s2 += red[k][threadIdx.x];
    out[c] = s2;
  }
}
inline cudaError_t reduce_rows(const float *part, int64_t n, int64_t stride, int64_t cols, float *out,
                               cudaStream_t st) {
  reduce_rows_kernel<<<(unsigned)((cols + 31) / 32), dim3(32, 32), 0, st>>>(part, n, stride, cols, out);
  return cudaGetLastError();
}

// =========================================================== short_conv ====
// A thread owns a run of tokens of one batch row and a vector of channels:
// the forward 8 channels (16 bytes of bf16) and TF tokens, the backward 4
// channels and TB tokens.  Every load of the run (the Kc-1 tokens before it,
// and in the backward the Kc-1 after it) is issued before any arithmetic,
// and the runs are unrolled at compile time, so the tap windows are
// registers renamed from token to token.  Document starts are one bit per
// token of the run: a tap reads zero when a document starts after the token
// it reads and at or before the token it feeds.
constexpr int CF_THREADS = 128, NCF = 8;
constexpr int CB_X = 16, CB_Y = 16, NCB = 4, TB = 8, CB_RUNS = 2;  // a CTA: 64 channels x 512 tokens

// N-element vector of T, loaded raw and widened to fp32.
template <typename T, int N> struct Raw;
template <> struct Raw<__nv_bfloat16, 8> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = __ldg(reinterpret_cast<const uint4 *>(p)); }
  __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};
template <> struct Raw<float, 8> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = __ldg(reinterpret_cast<const float4 *>(p));
    b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};
template <> struct Raw<__nv_bfloat16, 4> {
  uint2 u;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = __ldg(reinterpret_cast<const uint2 *>(p)); }
  __device__ __forceinline__ void zero() { u = make_uint2(0, 0); }
  __device__ __forceinline__ void get(float (&v)[4]) const {
    v[0] = __uint_as_float(u.x << 16);
    v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16);
    v[3] = __uint_as_float(u.y & 0xffff0000u);
  }
};
template <> struct Raw<float, 4> {
  float4 a;
  __device__ __forceinline__ void load(const float *p) { a = __ldg(reinterpret_cast<const float4 *>(p)); }
  __device__ __forceinline__ void zero() { a = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&v)[4]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  }
};
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float (&v)[4]) {
  *reinterpret_cast<uint2 *>(p) = make_uint2(pk(v[0], v[1]), pk(v[2], v[3]));
}
__device__ __forceinline__ void st4(float *p, const float (&v)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

// Bit j: token ta + j (j < n) starts a document (its row's first token, or
// its segment id differs from the previous token's); tokens past the row
// end count as starts (nothing reads across them).
__device__ __forceinline__ uint32_t doc_starts(const int32_t *seg, int64_t rowbase, int64_t T_, int64_t ta, int n) {
  uint32_t m = 0;
  for (int j = 0; j < n; ++j) {
    const int64_t t = ta + j;
    const bool st = t <= 0 || t >= T_ || (seg && seg[rowbase + t] != seg[rowbase + t - 1]);
    m |= (uint32_t)st << j;
  }
  return m;
}

// tokens per forward thread: 16 for bf16 (16-byte vectors), 8 for fp32
template <typename T> struct ConvTok { static constexpr int value = 16; };
template <> struct ConvTok<float> { static constexpr int value = 8; };

template <typename T, int KC>
__global__ void __launch_bounds__(CF_THREADS)
    short_conv_fwd_kernel(const T *__restrict__ x, const float *__restrict__ w, const float *__restrict__ bias,
                          const int32_t *__restrict__ seg, T *__restrict__ y, int64_t T_, int64_t D, int act) {
  constexpr int TF = ConvTok<T>::value, NW = TF + KC - 1;  // run and window tokens
  const int64_t c0 = ((int64_t)blockIdx.x * CF_THREADS + threadIdx.x) * NCF;
  if (c0 >= D) return;
  const int64_t b = blockIdx.z, t0 = (int64_t)blockIdx.y * TF, ta = t0 - (KC - 1);
  const T *xr = x + (b * T_ + ta) * D + c0;  // token ta (may lie before the row: never read there)
  Raw<T, NCF> raw[NW];
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    const int64_t t = ta + i;
    if (t >= 0 && t < T_)
      raw[i].load(xr + (int64_t)i * D);
    else
      raw[i].zero();
  }
  float wv[KC][NCF], bv[NCF];
#pragma unroll
  for (int k = 0; k < KC; ++k)
#pragma unroll
    for (int i = 0; i < NCF; ++i) wv[k][i] = w[k * D + c0 + i];
#pragma unroll
  for (int i = 0; i < NCF; ++i) bv[i] = bias ? bias[c0 + i] : 0.f;
  const uint32_t st = doc_starts(seg, b * T_, T_, ta, NW);
  T *yr = y + (b * T_ + t0) * D + c0;
#pragma unroll
  for (int i = 0; i < TF; ++i) {
    if (t0 + i >= T_) break;
    float a[NCF];
#pragma unroll
    for (int e = 0; e < NCF; ++e) a[e] = bv[e];
    // tap k reads window token i + k; blocked by a start in (i + k, i + KC - 1]
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const uint32_t between = ((1u << (KC - 1 - k)) - 1u) << (i + k + 1);
      if (!(st & between)) {
        float xv[NCF];
        raw[i + k].get(xv);
#pragma unroll
        for (int e = 0; e < NCF; ++e) a[e] += wv[k][e] * xv[e];
      }
    }
    if (act)
#pragma unroll
      for (int e = 0; e < NCF; ++e) a[e] *= sigm(a[e]);
    st8(yr + (int64_t)i * D, a);
  }
}

// Backward.  part: [B * gridDim.y][KC + 1][D] partial dW (taps 0..KC-1) and db.
// A CTA is CB_X x CB_Y threads: CB_X channel vectors by CB_Y token runs, each
// thread walking CB_RUNS runs of TB tokens (runs y, y + CB_Y, ...).
template <typename T, int KC>
__global__ void __launch_bounds__(CB_X *CB_Y)
    short_conv_bwd_kernel(const T *__restrict__ x, const float *__restrict__ w, const float *__restrict__ bias,
                          const int32_t *__restrict__ seg, const T *__restrict__ dy, T *__restrict__ dx,
                          float *__restrict__ part, int64_t T_, int64_t D, int act) {
  constexpr int NX = TB + 2 * (KC - 1), NG = TB + KC - 1;  // x window and dy / dz tokens
  __shared__ float red[CB_Y][KC + 1][CB_X * NCB];
  const int64_t c0 = ((int64_t)blockIdx.x * CB_X + threadIdx.x) * NCB;
  const bool on = c0 < D;
  const int64_t b = blockIdx.z;
  float acc[KC + 1][NCB];
#pragma unroll
  for (int k = 0; k <= KC; ++k)
#pragma unroll
    for (int e = 0; e < NCB; ++e) acc[k][e] = 0.f;
  float wv[KC][NCB], bv[NCB];
#pragma unroll
  for (int k = 0; k < KC; ++k)
#pragma unroll
    for (int e = 0; e < NCB; ++e) wv[k][e] = on ? w[k * D + c0 + e] : 0.f;
#pragma unroll
  for (int e = 0; e < NCB; ++e) bv[e] = (on && bias) ? bias[c0 + e] : 0.f;
  for (int run = 0; run < CB_RUNS; ++run) {
    const int64_t t0 = (((int64_t)blockIdx.y * CB_RUNS + run) * CB_Y + threadIdx.y) * TB;
    if (!on || t0 >= T_) continue;
    const int64_t ta = t0 - (KC - 1);  // first x token of the window
    const T *xr = x + (b * T_ + ta) * D + c0;
    const T *gr = dy + (b * T_ + t0) * D + c0;
    Raw<T, NCB> rx[NX], rg[NG];
#pragma unroll
    for (int i = 0; i < NX; ++i) {
      const int64_t t = ta + i;
      if (t >= 0 && t < T_)
        rx[i].load(xr + (int64_t)i * D);
      else
        rx[i].zero();
    }
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      if (t0 + i < T_)
        rg[i].load(gr + (int64_t)i * D);
      else
        rg[i].zero();
    }
    // starts of the x window's tokens (ta .. ta + NX - 1)
    const uint32_t st = doc_starts(seg, b * T_, T_, ta, NX);
    // dz of tokens t0 .. t0 + NG - 1 (window index i + KC - 1); zero past the row
    float dz[NG][NCB];
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      float a[NCB], gv[NCB];
#pragma unroll
      for (int e = 0; e < NCB; ++e) a[e] = bv[e];
#pragma unroll
      for (int k = 0; k < KC; ++k) {
        const uint32_t between = ((1u << (KC - 1 - k)) - 1u) << (i + k + 1);
        if (!(st & between)) {
          float xv[NCB];
          rx[i + k].get(xv);
#pragma unroll
          for (int e = 0; e < NCB; ++e) a[e] += wv[k][e] * xv[e];
        }
      }
      rg[i].get(gv);
#pragma unroll
      for (int e = 0; e < NCB; ++e) {
        if (act) {
          const float s = sigm(a[e]);
          dz[i][e] = gv[e] * s * (1.f + a[e] * (1.f - s));
        } else {
          dz[i][e] = gv[e];
        }
      }
      // dW, db of the run's own tokens: tap k of token i read window token i + k
      if (i < TB && t0 + i < T_) {
#pragma unroll
        for (int k = 0; k < KC; ++k) {
          const uint32_t between = ((1u << (KC - 1 - k)) - 1u) << (i + k + 1);
          if (!(st & between)) {
            float xv[NCB];
            rx[i + k].get(xv);
#pragma unroll
            for (int e = 0; e < NCB; ++e) acc[k][e] += xv[e] * dz[i][e];
          }
        }
#pragma unroll
        for (int e = 0; e < NCB; ++e) acc[KC][e] += dz[i][e];
      }
    }
    // dx_t = sum_k w_k dz_{t + KC-1-k} over the same document: token i of the
    // run (window index i + KC - 1) reaches dz_{i + j} (j = KC-1-k) unless a
    // document starts in (i + KC - 1, i + KC - 1 + j]
    T *dxr = dx + (b * T_ + t0) * D + c0;
#pragma unroll
    for (int i = 0; i < TB; ++i) {
      if (t0 + i >= T_) break;
      float o[NCB];
#pragma unroll
      for (int e = 0; e < NCB; ++e) o[e] = 0.f;
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        const uint32_t between = ((1u << j) - 1u) << (i + KC);
        if (!(st & between) && t0 + i + j < T_)
#pragma unroll
          for (int e = 0; e < NCB; ++e) o[e] += wv[KC - 1 - j][e] * dz[i + j][e];
      }
      st4(dxr + (int64_t)i * D, o);
    }
  }
#pragma unroll
  for (int k = 0; k <= KC; ++k)
#pragma unroll
    for (int e = 0; e < NCB; ++e) red[threadIdx.y][k][threadIdx.x * NCB + e] = acc[k][e];
  __syncthreads();
  const int64_t prow = b * gridDim.y + blockIdx.y;
  const int tid = threadIdx.y * CB_X + threadIdx.x;
  const int64_t cbase = (int64_t)blockIdx.x * CB_X * NCB;
  for (int e = tid; e < (KC + 1) * CB_X * NCB; e += CB_X * CB_Y) {
    const int k = e / (CB_X * NCB), c = e % (CB_X * NCB);
    if (cbase + c < D) {
      float s2 = 0.f;
#pragma unroll
      for (int yy = 0; yy < CB_Y; ++yy) s2 += red[yy][k][c];
      part[(prow * (KC + 1) + k) * D + cbase + c] = s2;
    }
  }
}

inline bool al16(const void *p) { return ((uintptr_t)p & 15) == 0; }
inline int log2_lanes(int64_t V) {
  switch (V) {
    case 8: return 0;
    case 16: return 1;
    case 32: return 2;
    case 64: return 3;
    case 128: return 4;
    case 256: return 5;
  }
  return -1;
}

}  // namespace fuse
}  // namespace glacore

using namespace glacore;
using namespace glacore::fuse;

static glacore_status cuda_st(cudaError_t e) { return status_of(e); }

extern "C" {

size_t norm_gate_bwd_workspace_size(int64_t rows, int64_t V) {
  if (rows < 0 || log2_lanes(V) < 0) return 0;
  return (size_t)ng_blocks(rows, V) * (size_t)V * sizeof(float);
}

glacore_status norm_gate_fwd(const void *o, const void *z, const float *w, int64_t rows, int64_t V, int32_t dtype,
                             float eps, void *y, glacore_stream_t stream) {
  const int lg = log2_lanes(V);
  if (rows < 0 || lg < 0 || (dtype != GLACORE_BF16 && dtype != GLACORE_F32) || !(eps >= 0.f))
    return GLACORE_ERR_INVALID_ARG;
  if (rows == 0) return GLACORE_OK;
  if (!o || !z || !w || !y || !al16(o) || !al16(z) || !al16(y)) return GLACORE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const int blocks = (int)ng_blocks(rows, V);
  if (dtype == GLACORE_BF16)
    norm_gate_fwd_kernel<__nv_bfloat16><<<blocks, NG_THREADS, 0, st>>>(
        (const __nv_bfloat16 *)o, (const __nv_bfloat16 *)z, w, (__nv_bfloat16 *)y, rows, (int)V, lg, eps);
  else
    norm_gate_fwd_kernel<float><<<blocks, NG_THREADS, 0, st>>>((const float *)o, (const float *)z, w, (float *)y,
                                                               rows, (int)V, lg, eps);
  mark_launch("norm_gate_fwd", st);
  return cuda_st(cudaGetLastError());
}

glacore_status norm_gate_bwd(const void *o, const void *z, const float *w, const void *dy, int64_t rows, int64_t V,
                             int32_t dtype, float eps, void *do_, void *dz, float *dw, void *workspace,
                             size_t workspace_bytes, glacore_stream_t stream) {
  const int lg = log2_lanes(V);
  if (rows < 0 || lg < 0 || (dtype != GLACORE_BF16 && dtype != GLACORE_F32) || !(eps >= 0.f) || !dw)
    return GLACORE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (rows == 0) return cuda_st(cudaMemsetAsync(dw, 0, (size_t)V * sizeof(float), st));
  if (!o || !z || !w || !dy || !do_ || !dz || !al16(o) || !al16(z) || !al16(dy) || !al16(do_) || !al16(dz))
    return GLACORE_ERR_INVALID_ARG;
  const size_t need = norm_gate_bwd_workspace_size(rows, V);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return GLACORE_ERR_WORKSPACE;
  const int blocks = (int)ng_blocks(rows, V);
  float *part = (float *)workspace;
  if (dtype == GLACORE_BF16)
    norm_gate_bwd_kernel<__nv_bfloat16><<<blocks, NG_THREADS, 0, st>>>(
        (const __nv_bfloat16 *)o, (const __nv_bfloat16 *)z, w, (const __nv_bfloat16 *)dy, (__nv_bfloat16 *)do_,
        (__nv_bfloat16 *)dz, part, rows, (int)V, lg, eps);
  else
    norm_gate_bwd_kernel<float><<<blocks, NG_THREADS, 0, st>>>((const float *)o, (const float *)z, w,
                                                               (const float *)dy, (float *)do_, (float *)dz, part,
                                                               rows, (int)V, lg, eps);
  mark_launch("norm_gate_bwd", st);
  if (const cudaError_t le = cudaGetLastError()) return cuda_st(le);
  const cudaError_t e = reduce_rows(part, blocks, V, V, dw, st);
  mark_launch("norm_gate_dw", st);
  return cuda_st(e);
}

size_t short_conv_bwd_workspace_size(int64_t B, int64_t T, int64_t D, int32_t Kc) {
  if (B < 1 || T < 0 || D < 8 || (D & 7) || Kc < 1 || Kc > 4) return 0;
  const int64_t per = (int64_t)CB_Y * CB_RUNS * TB;
  const int64_t ty = (T + per - 1) / per;
  return (size_t)(B * ty) * (size_t)(Kc + 1) * (size_t)D * sizeof(float);
}

glacore_status short_conv_fwd(const void *x, const float *w, const float *b, const int32_t *segment_ids, int64_t B,
                              int64_t T, int64_t D, int32_t Kc, int32_t dtype, int32_t activation, void *y,
                              glacore_stream_t stream) {
  if (B < 1 || T < 0 || D < 8 || (D & 7) || Kc < 1 || Kc > 4 || (activation != 0 && activation != 1) ||
      (dtype != GLACORE_BF16 && dtype != GLACORE_F32) || B > 65535)
    return GLACORE_ERR_INVALID_ARG;
  if (T == 0) return GLACORE_OK;
  if (!x || !w || !y || !al16(x) || !al16(y)) return GLACORE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const int tf = dtype == GLACORE_BF16 ? ConvTok<__nv_bfloat16>::value : ConvTok<float>::value;
  const dim3 grid((unsigned)((D / NCF + CF_THREADS - 1) / CF_THREADS), (unsigned)((T + tf - 1) / tf), (unsigned)B);
  if (grid.y > 65535u) return GLACORE_ERR_INVALID_ARG;
#define GLACORE_CONV_FWD(TY, KV)                                                                             \
  short_conv_fwd_kernel<TY, KV><<<grid, CF_THREADS, 0, st>>>((const TY *)x, w, b, segment_ids, (TY *)y, T, D, \
                                                              activation)
  if (dtype == GLACORE_BF16) {
    switch (Kc) {
      case 1: GLACORE_CONV_FWD(__nv_bfloat16, 1); break;
      case 2: GLACORE_CONV_FWD(__nv_bfloat16, 2); break;
      case 3: GLACORE_CONV_FWD(__nv_bfloat16, 3); break;
      default: GLACORE_CONV_FWD(__nv_bfloat16, 4); break;
    }
  } else {
    switch (Kc) {
      case 1: GLACORE_CONV_FWD(float, 1); break;
      case 2: GLACORE_CONV_FWD(float, 2); break;
      case 3: GLACORE_CONV_FWD(float, 3); break;
      default: GLACORE_CONV_FWD(float, 4); break;
    }
  }
#undef GLACORE_CONV_FWD
  mark_launch("short_conv_fwd", st);
  return cuda_st(cudaGetLastError());
}

glacore_status short_conv_bwd(const void *x, const float *w, const float *b, const int32_t *segment_ids,
                              const void *dy, int64_t B, int64_t T, int64_t D, int32_t Kc, int32_t dtype,
                              int32_t activation, void *dx, float *dw, float *db, void *workspace,
                              size_t workspace_bytes, glacore_stream_t stream) {
  if (B < 1 || T < 0 || D < 8 || (D & 7) || Kc < 1 || Kc > 4 || (activation != 0 && activation != 1) ||
      (dtype != GLACORE_BF16 && dtype != GLACORE_F32) || B > 65535 || !dw || !db)
    return GLACORE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (T == 0) {
    if (cudaMemsetAsync(dw, 0, (size_t)Kc * D * sizeof(float), st) != cudaSuccess) return GLACORE_ERR_CUDA;
    return cuda_st(cudaMemsetAsync(db, 0, (size_t)D * sizeof(float), st));
  }
  if (!x || !w || !dy || !dx || !al16(x) || !al16(dy) || !al16(dx)) return GLACORE_ERR_INVALID_ARG;
  const size_t need = short_conv_bwd_workspace_size(B, T, D, Kc);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace & 255)) return GLACORE_ERR_WORKSPACE;
  const int64_t per = (int64_t)CB_Y * CB_RUNS * TB;
  const dim3 grid((unsigned)((D / NCB + CB_X - 1) / CB_X), (unsigned)((T + per - 1) / per), (unsigned)B);
  const dim3 block(CB_X, CB_Y);
  float *part = (float *)workspace;
#define GLACORE_CONV_BWD(TY, KV)                                                                        \
  short_conv_bwd_kernel<TY, KV><<<grid, block, 0, st>>>((const TY *)x, w, b, segment_ids, (const TY *)dy, \
                                                         (TY *)dx, part, T, D, activation)
  if (dtype == GLACORE_BF16) {
    switch (Kc) {
      case 1: GLACORE_CONV_BWD(__nv_bfloat16, 1); break;
      case 2: GLACORE_CONV_BWD(__nv_bfloat16, 2); break;
      case 3: GLACORE_CONV_BWD(__nv_bfloat16, 3); break;
      default: GLACORE_CONV_BWD(__nv_bfloat16, 4); break;
    }
  } else {
    switch (Kc) {
      case 1: GLACORE_CONV_BWD(float, 1); break;
      case 2: GLACORE_CONV_BWD(float, 2); break;
      case 3: GLACORE_CONV_BWD(float, 3); break;
      default: GLACORE_CONV_BWD(float, 4); break;
    }
  }
#undef GLACORE_CONV_BWD
  mark_launch("short_conv_bwd", st);
  if (const cudaError_t le = cudaGetLastError()) return cuda_st(le);
  // dW rows 0..Kc-1 then db: partial rows of (Kc + 1) x D, summed in row order
  const int64_t nrows = B * (int64_t)grid.y;
  cudaError_t e = reduce_rows(part, nrows, (int64_t)(Kc + 1) * D, (int64_t)Kc * D, dw, st);
  if (e == cudaSuccess) e = reduce_rows(part + (int64_t)Kc * D, nrows, (int64_t)(Kc + 1) * D, D, db, st);
  mark_launch("short_conv_dw", st);
  return cuda_st(e);
}

}  // extern "C"
