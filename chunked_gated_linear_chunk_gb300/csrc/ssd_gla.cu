// ssd_gla.cu -- Mamba-2 SSD (scalar log-decay per head, B/C shared by a
// group of heads) through the GLA tensor-core kernels.
//
// SSD is GLA with every key channel of a head carrying the same gate (FLAT
// blog, "Gated Linear Attention" / "Mamba-2": the per-head decay is the
// scalar special case of the per-channel decay): with g_gla[t,h,c] =
// g_ssd[t,h] for all c the recurrences coincide,
//   S_t = exp(g_t) S_{t-1} + k_t v_t^T,   o_t = scale S_t^T q_t.
// The tensor-core kernels read q and k of a head's group, the per-head gate
// and the V-column v and do in place (their grouped-head and per-head-gate
// modes; v's and do's columns past V read as zeros), and write o and dv in
// place.  These kernels pad h0 and dht to V = 128 and cut the final state and
// dh0 back, and map the GLA gradients back: dq and dk summed over the heads
// that share q and k, dg summed over K (the gradient of a gate shared by K
// channels).
#include "internal.cuh"

namespace glacore {
namespace ssdx {

constexpr int KX = 128, VX = 128;

// states [n*H, K, V] <-> [n*H, K, 128] (pad with zeros / cut)
__global__ void pad_state_kernel(int64_t mats, int64_t V, const float *src, float *dst) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // element of dst
  if (i >= mats * KX * VX) return;
  const int64_t c = i % VX, rowk = i / VX;
  dst[i] = c < V ? src[rowk * V + c] : 0.f;
}
__global__ void cut_state_kernel(int64_t mats, int64_t V, const float *src, float *dst) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // element of dst
  if (i >= mats * KX * V) return;
  const int64_t c = i % V, rowk = i / V;
  dst[i] = src[rowk * VX + c];
}
// dq / dk: sum over the G = H / Hqk heads of a group, fp32, rounded once.
// One thread per (token, group, 8 channels).
__global__ void reduce_heads_kernel(int64_t BT, int64_t H, int64_t Hqk, const uint4 *x, uint4 *out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BT * Hqk * (KX / 8)) return;
  const int64_t c8 = i % (KX / 8), tq = i / (KX / 8), t = tq / Hqk, hq = tq - t * Hqk;
  const int64_t G = H / Hqk;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int64_t j = 0; j < G; ++j) {
    const uint4 w = x[((t * H + hq * G + j) * (KX / 8)) + c8];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc[2 * e] += __uint_as_float(u[e] << 16);
      acc[2 * e + 1] += __uint_as_float(u[e] & 0xffff0000u);
    }
  }
  uint32_t r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
    r[e] = *reinterpret_cast<uint32_t *>(&p);
  }
  out[i] = make_uint4(r[0], r[1], r[2], r[3]);
}
// dg[t,h] = sum over the K channels; one warp per (token, head)
__global__ void sum_channels_kernel(int64_t rows, const float4 *x, float *dg) {
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float4 a = x[row * (KX / 4) + lane];
  float s = (a.x + a.y) + (a.z + a.w);
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) dg[row] = s;
}

static unsigned blocks_of(int64_t n, int per) { return (unsigned)((n + per - 1) / per); }

cudaError_t pad_states(int64_t mats, int64_t V, const float *src, float *dst, cudaStream_t st) {
  pad_state_kernel<<<blocks_of(mats * KX * VX, 256), 256, 0, st>>>(mats, V, src, dst);
  mark_launch("ssd_pad_state", st);
  return cudaGetLastError();
}
cudaError_t cut_states(int64_t mats, int64_t V, const float *src, float *dst, cudaStream_t st) {
  cut_state_kernel<<<blocks_of(mats * KX * V, 256), 256, 0, st>>>(mats, V, src, dst);
  mark_launch("ssd_cut_state", st);
  return cudaGetLastError();
}
cudaError_t reduce_heads(int64_t BT, int64_t H, int64_t Hqk, const void *x, void *out, cudaStream_t st) {
  reduce_heads_kernel<<<blocks_of(BT * Hqk * (KX / 8), 256), 256, 0, st>>>(BT, H, Hqk, (const uint4 *)x,
                                                                          (uint4 *)out);
  mark_launch("ssd_reduce_heads", st);
  return cudaGetLastError();
}
cudaError_t sum_channels(int64_t rows, const float *x, float *dg, cudaStream_t st) {
  sum_channels_kernel<<<blocks_of(rows, 8), 256, 0, st>>>(rows, (const float4 *)x, dg);
  mark_launch("ssd_sum_channels", st);
  return cudaGetLastError();
}

}  // namespace ssdx
}  // namespace glacore
