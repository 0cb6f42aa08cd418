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

// ---- per-chunk gate slot, shared by the SSD kernels --------------------
namespace gsl {
constexpr int NG = 3;
constexpr uint32_t GSLOT = 7680;
// gate slot (floats):
//   EG [0, 64)      scale exp(G_t) (0 past the chunk's end)
//   EGR [64, 128)   exp(Gam - G_s) (0 past the end)
//   B [128, 192)    exp(G_r - G_s), r the last token of s's 16-token block
//   EGAM at 192     exp(Gam)
//   A [196, 452)    row t, block b < t / 16: scale exp(G_t - G_r), r the
//                   last token of block b (4 per row)
//   G [452, 516)    G
//   DD [516, 1796)  diagonal blocks: [4][16][20], scale exp(G_t - G_s) for
//                   s <= t in the same block, 0 above (row stride 20), as
//                   products of the per-token factors exp(g)
//   E [1796, 1860)  exp(g_t)
// Off the diagonal, exp(G_t - G_s) = exp(G_t - G_r) exp(G_r - G_s) with
// t > r >= s: both factors in (0, 1].
constexpr int G_EG = 0, G_EGR = 64, G_B = 128, G_EGAM = 192, G_A = 196, G_G = 452, G_DD = 516, G_E = 1796;
}  // namespace gsl

using namespace tc;

// The decayed causal P of one chunk as bf16 tiles (K-major A of a product
// with P on the left; with HILO as hi / lo tiles, hi = bf16(P) and
// lo = bf16(P - hi)):  P[t,s] = X[t,s] F[t,s], F = scale exp(G_t - G_s) for
// s <= t, else 0, from the gate slot's factor tables, X the C x C product
// in TMEM (q k^T, or do v^T in the backward).  The M = 64
// accumulator holds warp qw's rows 16 qw .. 16 qw + 15 in lanes 0..15;
// lanes 16..31 take the second 16-column block of each pair (shuffled
// over), so every lane writes one block.  Blocks above the diagonal stay
// zero (written once by mask_tile_init).
template <bool HILO>
__device__ __forceinline__ void decay_mask(uint32_t t_acc, uint32_t lane_off, int qw, int lane, uint8_t *hi,
                                           uint8_t *lo, const float *gs) {
  using namespace gsl;
  const int rl = lane & 15, row = qw * 16 + rl;
  const bool second = lane >= 16;
  uint32_t r[2][16], x[2][16];
#pragma unroll
  for (int cp = 0; cp < 4; cp += 2)
    if (cp <= qw) {
      tmem_ld16(t_acc + lane_off + cp * 16, r[cp / 2]);
      tmem_ld16(t_acc + lane_off + cp * 16 + 16, x[cp / 2]);
    }
  tmem_ld_wait(r[0]);
  tmem_tie(x[0]);
  if (qw >= 2) {
    tmem_tie(r[1]);
    tmem_tie(x[1]);
  }
  const uint32_t ga = smem_u32(gs);
  const float4 arow = lds_f4(ga + 4u * (G_A + 4 * row));
#pragma unroll
  for (int cp = 0; cp < 4; cp += 2) {
    if (cp <= qw) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t sh = __shfl_sync(0xffffffffu, x[cp / 2][i], rl);
        v[i] = __uint_as_float(second ? sh : r[cp / 2][i]);
      }
      const int cb = cp + (second ? 1 : 0);
      if (cb <= qw) {
        float f[16];
        if (cb < qw) {
          const float a = cb == 0 ? arow.x : (cb == 1 ? arow.y : arow.z);
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 b = lds_f4(ga + 4u * (G_B + cb * 16 + i));
            f[i] = a * b.x;
            f[i + 1] = a * b.y;
            f[i + 2] = a * b.z;
            f[i + 3] = a * b.w;
          }
        } else {
          const uint32_t dd = ga + 4u * (G_DD + (qw * 16 + rl) * 20);
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 b = lds_f4(dd + 4u * i);
            f[i] = b.x;
            f[i + 1] = b.y;
            f[i + 2] = b.z;
            f[i + 3] = b.w;
          }
        }
        uint32_t w[8], wl[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x0 = v[2 * e] * f[2 * e], x1 = v[2 * e + 1] * f[2 * e + 1];
          w[e] = pack_bf16(x0, x1);
          if (HILO) wl[e] = pack_bf16(x0 - __uint_as_float(w[e] << 16), x1 - __uint_as_float(w[e] & 0xffff0000u));
        }
        const uint32_t o0 = sw128_off(row, cb * 16, 64), o1 = sw128_off(row, cb * 16 + 8, 64);
        st_shared_v4(smem_u32(hi + o0), w[0], w[1], w[2], w[3]);
        st_shared_v4(smem_u32(hi + o1), w[4], w[5], w[6], w[7]);
        if (HILO) {
          st_shared_v4(smem_u32(lo + o0), wl[0], wl[1], wl[2], wl[3]);
          st_shared_v4(smem_u32(lo + o1), wl[4], wl[5], wl[6], wl[7]);
        }
      }
    }
  }
}

// decay_mask<false> in two steps, so that the tile can be computed while
// the products that read the previous tile are still running: the packed
// bf16 words of the lane's two 16-column blocks (2 k, plus 1 for lanes
// 16..31, k = 0, 1; valid where the block is at or below the diagonal) ...
__device__ __forceinline__ void decay_tile_regs(uint32_t t_acc, uint32_t lane_off, int qw, int lane, const float *gs,
                                                uint32_t (&w)[2][8]) {
  using namespace gsl;
  const int rl = lane & 15, row = qw * 16 + rl;
  const bool second = lane >= 16;
  const uint32_t ga = smem_u32(gs);
  const float4 arow = lds_f4(ga + 4u * (G_A + 4 * row));
#pragma unroll
  for (int cp = 0; cp < 4; cp += 2) {
    if (cp <= qw) {
      uint32_t r0[16], r1[16];
      tmem_ld16(t_acc + lane_off + cp * 16, r0);
      tmem_ld16(t_acc + lane_off + cp * 16 + 16, r1);
      tmem_ld_wait(r0);
      tmem_tie(r1);
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t sh = __shfl_sync(0xffffffffu, r1[i], rl);
        v[i] = __uint_as_float(second ? sh : r0[i]);
      }
      const int cb = cp + (second ? 1 : 0);
      float f[16];
      if (cb < qw) {
        const float a = cb == 0 ? arow.x : (cb == 1 ? arow.y : arow.z);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 b = lds_f4(ga + 4u * (G_B + cb * 16 + i));
          f[i] = a * b.x;
          f[i + 1] = a * b.y;
          f[i + 2] = a * b.z;
          f[i + 3] = a * b.w;
        }
      } else {
        const uint32_t dd = ga + 4u * (G_DD + (qw * 16 + rl) * 20);
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 b = lds_f4(dd + 4u * i);
          f[i] = b.x;
          f[i + 1] = b.y;
          f[i + 2] = b.z;
          f[i + 3] = b.w;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) w[cp / 2][e] = pack_bf16(v[2 * e] * f[2 * e], v[2 * e + 1] * f[2 * e + 1]);
    }
  }
}
// ... and their store into the tile.
__device__ __forceinline__ void decay_tile_store(uint8_t *tile, int qw, int lane, const uint32_t (&w)[2][8]) {
  const int rl = lane & 15, row = qw * 16 + rl;
  const int sb = lane >= 16 ? 1 : 0;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int cb = 2 * k + sb;
    if (2 * k <= qw && cb <= qw) {
      st_shared_v4(smem_u32(tile + sw128_off(row, cb * 16, 64)), w[k][0], w[k][1], w[k][2], w[k][3]);
      st_shared_v4(smem_u32(tile + sw128_off(row, cb * 16 + 8, 64)), w[k][4], w[k][5], w[k][6], w[k][7]);
    }
  }
}

// Row c (channel) of the bf16 state tile (128 rows x 64 columns, 128-byte
// swizzle): the B operand of q S, MN-major.
__device__ __forceinline__ void store_state_row(uint8_t *St, int c, const float (&S)[64]) {
#pragma unroll
  for (int n = 0; n < 64; n += 8)
    st_shared_v4(smem_u32(St + sw128_off(c, n, 128)), pack_bf16(S[n], S[n + 1]), pack_bf16(S[n + 2], S[n + 3]),
                 pack_bf16(S[n + 4], S[n + 5]), pack_bf16(S[n + 6], S[n + 7]));
}

__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t x, float f) {
  return pack_bf16(__uint_as_float(x << 16) * f, __uint_as_float(x & 0xffff0000u) * f);
}

// The gate slot of one chunk, built by 64 threads (two warps; thread t
// owns token t; named barrier `bar` over those 64 threads).  gt is token
// t's log-decay (0 past the chunk's end L).  Returns exp(Gam - G_t) in egr
// and scale exp(G_t) in eg (both 0 past the end).  The decay factors of
// rows past the end are 0, so those rows of every decayed C x C tile are 0
// (the next document's tokens there add nothing).
__device__ __forceinline__ void gate_factors(float *gs, int t, int lane, int L, float scale, float gt, int bar,
                                             float &egr, float &eg) {
  using namespace gsl;
  const int blk = t >> 4, r = t & 15;
  // G: inclusive prefix sum over the chunk (the second warp adds the first's total)
  float Gt = gt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, Gt, o);
    if (lane >= o) Gt += y;
  }
  if (t == 31) gs[G_EGAM + 2] = Gt;
  named_bar(bar, 64);
  const uint32_t ga = smem_u32(gs);
  if (t >= 32) Gt += lds_f1(ga + 4u * (G_EGAM + 2));
  gs[G_G + t] = Gt;
  gs[G_E + t] = __expf(gt);
  if (t == L - 1) {
    gs[G_EGAM] = __expf(Gt);
    gs[G_EGAM + 1] = Gt;
  }
  named_bar(bar, 64);
  const float Gam = lds_f1(ga + 4u * (G_EGAM + 1));
  egr = t < L ? __expf(Gam - Gt) : 0.f;
  eg = t < L ? scale * __expf(Gt) : 0.f;
  gs[G_EG + t] = eg;
  gs[G_EGR + t] = egr;
  gs[G_B + t] = __expf(lds_f1(ga + 4u * (G_G + (t | 15))) - Gt);
  {  // row factors of row t (blocks before t's own)
    float av[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) av[b] = (b < blk && t < L) ? scale * __expf(Gt - lds_f1(ga + 4u * (G_G + 16 * b + 15))) : 0.f;
    *reinterpret_cast<float4 *>(gs + G_A + 4 * t) = make_float4(av[0], av[1], av[2], av[3]);
  }
  {  // row t of its diagonal block: scale exp(G_t - G_c) = scale prod_{c < i <= t} exp(g_i)
    const uint32_t e = ga + 4u * (G_E + 16 * blk);
    float ev[16];
#pragma unroll
    for (int c = 0; c < 16; c += 4) {
      const float4 x = lds_f4(e + 4u * c);
      ev[c] = x.x;
      ev[c + 1] = x.y;
      ev[c + 2] = x.z;
      ev[c + 3] = x.w;
    }
    float dv[16];
    float run = scale;
#pragma unroll
    for (int c = 15; c >= 0; --c) {
      dv[c] = (c <= r && t < L) ? run : 0.f;
      if (c <= r && c > 0) run *= ev[c];
    }
    float *dd = gs + G_DD + t * 20;
#pragma unroll
    for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4 *>(dd + i) = make_float4(dv[i], dv[i + 1], dv[i + 2], dv[i + 3]);
  }
}

// True when these kernels run the SSD problem: bf16, K = 128, V = 64, any
// head grouping, q / k / v token strides TMA can address, chunk 0 or 64.
bool supported(const glacore_problem *p);
// Scratch of the SSD kernels (launch order of packed documents; the
// backward's fp32 dq / dk accumulators and per-token gate-gradient terms).
size_t workspace_bytes(const glacore_problem *p, bool backward);
size_t bwd_workspace_bytes(const glacore_problem *p);
cudaError_t fwd(const Prob &pr, const Docs &docs, const glacore_problem *p, void *o, float *ht, char *ws,
                cudaStream_t st);
cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO, const float *dht,
                void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws, cudaStream_t st);

}  // namespace ssd
}  // namespace glacore
