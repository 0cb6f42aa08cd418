// tc_ssd_bwd.cu -- backward of the SSD tcgen05 path (forward formulas in
// tc_ssd.cuh).
//
// Per chunk, with S_in the state entering it, dS the gradient of the state
// leaving it, F = scale exp(G_t - G_s) (s <= t, else 0) and the forward's
// A = (q k^T) (.) F, o = scale diag(exp(G)) q S_in + A v
// (FLAT blog, "Backward Recurrence" for the reverse state-gradient walk and
// the gate gradient; the products below are the chunkwise form of it):
//
//   dA   = (do v^T) (.) F                                  (masked, decayed)
//   dq_h = scale diag(exp(G)) do S_in^T + dA k
//   dk_h = dA^T q + diag(exp(Gam - G)) v dS^T
//   dv   = A^T do + diag(exp(Gam - G)) k dS
//   dS  <- exp(Gam) dS + scale q^T diag(exp(G)) do        (entering the chunk)
//   dg_t = sum over the document's tokens m >= t of
//          (q_m . dq_h,m - k_m . dk_h,m)  +  <dht, S_T>
//
// (the last line: the log-decay g_t scales every state from t on, so its
// gradient collects the q.dq and k.dk terms of all later tokens and the
// final-state term).  dq_h, dk_h are one head's terms; q and k are shared by
// the heads of a group, so those are summed over the group's heads: every
// CTA adds its fp32 tiles into dq / dk accumulators with TMA reduce-add at
// L2, and one small kernel rounds them to bf16.
//
// Two launches, one CTA per (document, head), 512 threads each:
//   pass A walks the chunks in order: recomputes S (k^T vt, as the
//          forward), emits dq_h (reduce-add) and q . dq_h per token, and
//          <dht, S_T> per (document, head);
//   pass B walks them in reverse: carries dS, emits dv, dk_h (reduce-add)
//          and dg (the reverse sum, carried across chunks), and dh0.
#include "tc_ssd.cuh"

namespace glacore {
namespace ssd {

struct BwdMaps {
  CUtensorMap q, k, v, dout, dqa, dka;
};

struct BwdArgs {
  Units units;
  int64_t H;
  int32_t hq_div;
  float scale;
  const float *g;     // [BT, H]
  const float *h0;    // [n_docs, H, K, V] or null
  const float *dht;   // [n_docs, H, K, V] or null
  float *dh0;         // [n_docs, H, K, V] or null
  __nv_bfloat16 *dv;  // [BT, H, V]
  float *dg;          // [BT, H]
  float *qdq;         // [BT, H]: q . dq_h per token (pass A -> pass B)
  float *sdht;        // [n_docs, H]: <dht, S_T> (pass A -> pass B)
  int *err;
};

namespace pas {  // pass A shared memory (bytes)
constexpr int NS = 2;
constexpr uint32_t Q = 0;         // 2 x 16 KB
constexpr uint32_t K = 32768;     // 2 x 16 KB
constexpr uint32_t V = 65536;     // 2 x 8 KB
constexpr uint32_t DO = 81920;    // 2 x 8 KB
constexpr uint32_t VT = 98304;    // 2 x 8 KB: v (.) exp(Gam - G_s)
constexpr uint32_t DOT = 114688;  // 2 x 8 KB: do (.) scale exp(G_t)
constexpr uint32_t DAF = 131072;  // 2 x 8 KB: dA (bf16, K-major A of dA k)
constexpr uint32_t S = 147456;    // 2 x 16 KB: S as bf16
constexpr uint32_t DQT = 180224;  // 16 KB: 2 KB staging buffers, two per output warp
constexpr uint32_t GS = 196608;
constexpr uint32_t BYTES = GS + gsl::NG * gsl::GSLOT;
}  // namespace pas

namespace pbs {  // pass B shared memory (bytes)
constexpr int NS = 2;
constexpr uint32_t Q = 0;
constexpr uint32_t K = 32768;
constexpr uint32_t V = 65536;
constexpr uint32_t DO = 81920;
constexpr uint32_t VT = 98304;    // 2 x 8 KB
constexpr uint32_t DOT = 114688;  // 2 x 8 KB
constexpr uint32_t A = 131072;    // 8 KB: A (bf16)
constexpr uint32_t DAF = 139264;  // 8 KB: dA (bf16)
constexpr uint32_t DS = 147456;   // 2 x 16 KB: dS as bf16 (rows = channel)
constexpr uint32_t DKT = 180224;  // 16 KB: 2 KB staging buffers, two per output warp
constexpr uint32_t GS = 196608;
constexpr uint32_t BYTES = GS + gsl::NG * gsl::GSLOT;
}  // namespace pbs

// One warp's 16 rows (16 qw .. 16 qw + 15) of an M = 64 accumulator with
// 128 columns, read out of TMEM whole: y[r][i] is column 32 r + i of row
// 16 qw + (lane & 15) for lanes 0..15, column 32 r + 16 + i for lanes 16..31.
__device__ __forceinline__ void tmem_rows128(uint32_t t_acc, uint32_t lane_off, int lane, float (&y)[4][16]) {
  const int rl = lane & 15;
  const bool second = lane >= 16;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    uint32_t a0[16], a1[16];
    tmem_ld16(t_acc + lane_off + 32 * r, a0);
    tmem_ld16(t_acc + lane_off + 32 * r + 16, a1);
    tmem_ld_wait(a0);
    tmem_tie(a1);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t sh = __shfl_sync(0xffffffffu, a1[i], rl);
      y[r][i] = __uint_as_float(second ? sh : a0[i]);
    }
  }
}

// Adds those rows (y, as tmem_rows128 leaves them) of this CTA's 64 x 128
// fp32 tile of a per-head gradient into the group accumulator (map m: boxes
// of 32 channels x 16 rows; rows tok0 + 16 qw .., head group hq), by TMA
// reduce-add at L2, in four rounds of 32 channels through the warp's two
// 2 KB staging buffers (stg, used in turn: a buffer is rewritten once the
// reduce issued from it two rounds earlier has read it).  Rows at or past L
// are added as zeros.  Returns this lane's share of sum_c x[row, c] y[row, c],
// x the bf16 tile (q or k of the chunk: two 64-column blocks, 128-byte
// swizzle).
__device__ __forceinline__ float reduce_rows(const float (&y)[4][16], int qw, int lane, int L, uint8_t *stg,
                                             const uint8_t *xt, const CUtensorMap *m, int hq, int tok0) {
  const int rl = lane & 15, row = qw * 16 + rl;
  const bool second = lane >= 16, live = row < L;
  float dot = 0.f;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int c0 = 32 * r + (second ? 16 : 0);
#pragma unroll
    for (int i = 0; i < 16; i += 8) {
      const uint4 xv = lds_u4(smem_u32(xt) + sw128_off(row, c0 + i, 64));
      dot += __uint_as_float(xv.x << 16) * y[r][i] + __uint_as_float(xv.x & 0xffff0000u) * y[r][i + 1] +
             __uint_as_float(xv.y << 16) * y[r][i + 2] + __uint_as_float(xv.y & 0xffff0000u) * y[r][i + 3] +
             __uint_as_float(xv.z << 16) * y[r][i + 4] + __uint_as_float(xv.z & 0xffff0000u) * y[r][i + 5] +
             __uint_as_float(xv.w << 16) * y[r][i + 6] + __uint_as_float(xv.w & 0xffff0000u) * y[r][i + 7];
    }
    uint8_t *buf = stg + (r & 1) * 2048;
    if (lane == 0) bulk_wait_read_all_but_one();  // the reduce from this buffer, two rounds back
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const uint32_t off = sw128_off_f32(rl, (second ? 16 : 0) + i, 16);
      st_shared_v4(smem_u32(buf + off), __float_as_uint(live ? y[r][i] : 0.f), __float_as_uint(live ? y[r][i + 1] : 0.f),
                   __float_as_uint(live ? y[r][i + 2] : 0.f), __float_as_uint(live ? y[r][i + 3] : 0.f));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_reduce_add_3d(m, buf, 32 * r, hq, tok0 + 16 * qw);
      bulk_commit();
    }
  }
  return dot;
}

// Adds one warp's 16 rows (16 qw .. 16 qw + 15) of this CTA's 64 x 128
// fp32 tile of a per-head gradient (M = 64 accumulator t_acc, 128 columns)
// into the group accumulator (map m: boxes of 32 channels x 16 rows; rows
// tok0 + 16 qw .., head group hq), by TMA reduce-add at L2, in four rounds
// of 32 channels through the warp's two 2 KB staging buffers (stg, used in
// turn: a buffer is rewritten once the reduce issued from it two rounds
// earlier has read it).  Rows at or past L are added as zeros.  Returns
// this lane's share of sum_c x[row, c] acc[row, c], x the bf16 tile (q or
// k of the chunk: two 64-column blocks, 128-byte swizzle).  Lanes r and
// r + 16 share row 16 qw + r (the first and second 16 columns of a round).
__device__ __forceinline__ float reduce_warp_rows(uint32_t t_acc, uint32_t lane_off, int qw, int lane, int L,
                                                  uint8_t *stg, const uint8_t *xt, const CUtensorMap *m, int hq,
                                                  int tok0) {
  const int rl = lane & 15, row = qw * 16 + rl;
  const bool second = lane >= 16, live = row < L;
  float dot = 0.f;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    uint32_t a0[16], a1[16];
    tmem_ld16(t_acc + lane_off + 32 * r, a0);
    tmem_ld16(t_acc + lane_off + 32 * r + 16, a1);
    tmem_ld_wait(a0);
    tmem_tie(a1);
    float y[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t sh = __shfl_sync(0xffffffffu, a1[i], rl);
      y[i] = __uint_as_float(second ? sh : a0[i]);
    }
    const int c0 = 32 * r + (second ? 16 : 0);
#pragma unroll
    for (int i = 0; i < 16; i += 8) {
      const uint4 xv = lds_u4(smem_u32(xt) + sw128_off(row, c0 + i, 64));
      dot += __uint_as_float(xv.x << 16) * y[i] + __uint_as_float(xv.x & 0xffff0000u) * y[i + 1] +
             __uint_as_float(xv.y << 16) * y[i + 2] + __uint_as_float(xv.y & 0xffff0000u) * y[i + 3] +
             __uint_as_float(xv.z << 16) * y[i + 4] + __uint_as_float(xv.z & 0xffff0000u) * y[i + 5] +
             __uint_as_float(xv.w << 16) * y[i + 6] + __uint_as_float(xv.w & 0xffff0000u) * y[i + 7];
    }
    uint8_t *buf = stg + (r & 1) * 2048;
    if (lane == 0) bulk_wait_read_all_but_one();  // the reduce from this buffer, two rounds back
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
      const uint32_t off = sw128_off_f32(rl, (second ? 16 : 0) + i, 16);
      st_shared_v4(smem_u32(buf + off), __float_as_uint(live ? y[i] : 0.f), __float_as_uint(live ? y[i + 1] : 0.f),
                   __float_as_uint(live ? y[i + 2] : 0.f), __float_as_uint(live ? y[i + 3] : 0.f));
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_reduce_add_3d(m, buf, 32 * r, hq, tok0 + 16 * qw);
      bulk_commit();
    }
  }
  return dot;
}

// =========================================================================
// pass A: chunks in order
//   warp 0       TMA (q, k, v, do; 2 stages)
//   warp 1       MMA: dP = do v^T, U = k^T vt, dq_h = dot S_in^T + dA k
//   warps 2..5   mask: dA = dP (.) F (bf16)
//   warps 6..9   state: S (as the forward), <dht, S_T> at the end
//   warps 10..13 dq_h tile -> reduce-add, q . dq_h per token
//   warps 14, 15 gate: the gate slot, vt, dot = do (.) scale exp(G)
// TMEM: U[2] at 0/64, dP[2] at 128/192, DQ[2] at 256/384 (64 x 128 each).
// =========================================================================
__global__ void __launch_bounds__(512, 1) ssd_bwd_a_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using namespace pas;
  using namespace gsl;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[NS], empty[NS], gready[NG], gfree[NG], u_full[2], dp_full[2], dq_full[2], p_ready[2],
      s_ready[2], dq_free[2], drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float red[4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t H = a.H;
  const int h = (int)((int64_t)blockIdx.x % H);
  const int hq = a.hq_div > 1 ? h / a.hq_div : h;
  const int64_t u = a.units.at((int64_t)blockIdx.x / H);
  const Unit un = a.units.get(u);
  const int64_t d = un.doc, s0 = un.start, s1 = un.end;
  const int nch = (int)((s1 - s0 + C - 1) / C);
  auto chunk_tok = [&](int j) -> int64_t { return s0 + (int64_t)j * C; };
  auto chunk_len = [&](int j) -> int { return (int)min((int64_t)C, s1 - chunk_tok(j)); };
  auto slot_of = [&](int j) -> float * { return reinterpret_cast<float *>(sm + GS + (j % NG) * GSLOT); };

  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 129);  // the MMA commit and the 128 threads that read q
    }
    for (int i = 0; i < NG; ++i) {
      mbar_init(&gready[i], 64);
      mbar_init(&gfree[i], 256);  // mask and state warpgroups
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&u_full[i], 1);
      mbar_init(&dp_full[i], 1);
      mbar_init(&dq_full[i], 1);
      mbar_init(&p_ready[i], 128);
      mbar_init(&s_ready[i], 128);
      mbar_init(&dq_free[i], 128);
    }
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base, sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
#define SSD_FAIL                \
  {                             \
    atomicExch(&abort_flag, 1); \
    break;                      \
  }
  auto tU = [&](int b) { return tbase + 64u * b; };
  auto tDP = [&](int b) { return tbase + 128u + 64u * b; };
  auto tDQ = [&](int b) { return tbase + 256u + 128u * b; };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dout);
      int issued = 0;
      for (int j = 0; j < nch; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(&empty[s], ((j / NS) - 1) & 1, WAIT_CYCLES)) SSD_FAIL
        if (*abortp) break;
        const int tok = (int)chunk_tok(j);
        mbar_expect_tx(&full[s], 16384 + 16384 + 8192 + 8192);
        tma_load_3d(sm + Q + s * 16384, &maps.q, 0, hq, tok, &full[s]);
        tma_load_3d(sm + Q + s * 16384 + 8192, &maps.q, 64, hq, tok, &full[s]);
        tma_load_3d(sm + K + s * 16384, &maps.k, 0, hq, tok, &full[s]);
        tma_load_3d(sm + K + s * 16384 + 8192, &maps.k, 64, hq, tok, &full[s]);
        tma_load_3d(sm + V + s * 8192, &maps.v, 0, h, tok, &full[s]);
        tma_load_3d(sm + DO + s * 8192, &maps.dout, 0, h, tok, &full[s]);
        // the tiles of chunk j + 2 into L2 ahead of their load
        if (j + 2 < nch) {
          const int tp = (int)chunk_tok(j + 2);
          tma_prefetch_3d(&maps.q, 0, hq, tp);
          tma_prefetch_3d(&maps.q, 64, hq, tp);
          tma_prefetch_3d(&maps.k, 0, hq, tp);
          tma_prefetch_3d(&maps.k, 64, hq, tp);
          tma_prefetch_3d(&maps.v, 0, h, tp);
          tma_prefetch_3d(&maps.dout, 0, h, tp);
        }
        issued = j + 1;
      }
      for (int j = max(0, issued - NS); j < issued; ++j)
        if (!mbar_wait(&full[j % NS], (j / NS) & 1, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idDP = idesc_bf16(64, 64, false, false);
      constexpr uint32_t idU = idesc_bf16(128, 64, true, true);
      constexpr uint32_t idQ1 = idesc_bf16(64, 128, false, false);
      constexpr uint32_t idQ2 = idesc_bf16(64, 128, false, true);
      for (int j = 0; j < nch && !*abortp; ++j) {
        const int b = j & 1, s = j % NS;
        const uint32_t qa = sbase + Q + s * 16384, ka = sbase + K + s * 16384;
        (void)qa;
        // dP = do v^T (its buffer was read by the mask step of j - 2)
        if (!mbar_wait(&full[s], (j / NS) & 1, WAIT_CYCLES)) SSD_FAIL
        tc_fence_after();
        {
          const uint32_t da = sbase + DO + s * 8192, va = sbase + V + s * 8192;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tDP(b), kdesc(da, ks, 64), kdesc(va, ks, 64), idDP, ks);
          mma_commit(&dp_full[b]);
        }
        // U = k^T vt (its buffer was read by the state step of j - 2)
        if (!mbar_wait(&gready[j % NG], (j / NG) & 1, WAIT_CYCLES)) SSD_FAIL
        tc_fence_after();
        {
          const uint32_t vt = sbase + VT + b * 8192;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tU(b), mdesc(ka, ks, 8192), mdesc(vt, ks, 8192), idU, ks);
          mma_commit(&u_full[b]);
        }
        // dq_h = dot S_in^T + dA k
        if (!mbar_wait(&s_ready[(j + 1) & 1], (j >> 1) & 1, WAIT_CYCLES) ||
            !mbar_wait(&p_ready[b], (j >> 1) & 1, WAIT_CYCLES) ||
            (j >= 2 && !mbar_wait(&dq_free[b], ((j - 2) >> 1) & 1, WAIT_CYCLES)))
          SSD_FAIL
        tc_fence_after();
        {
          const uint32_t dot = sbase + DOT + b * 8192, Sa = sbase + S + ((j + 1) & 1) * 16384;
          const uint32_t daf = sbase + DAF + b * 8192;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tDQ(b), kdesc(dot, ks, 64), kdesc(Sa, ks, 128), idQ1, ks);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tDQ(b), kdesc(daf, ks, 64), mdesc(ka, ks, 8192), idQ2, 1);
          mma_commit(&dq_full[b]);
          mma_commit(&empty[s]);
        }
      }
      mma_commit(&drain);
      if (!mbar_wait(&drain, 0, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else if (warp < 6) {
    // ---------------- mask: dA = (do v^T) (.) F ----------------
    const int qw = warp & 3;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    for (int t = 0; t < 2; ++t) mask_tile_init(sm + DAF + t * 8192, qw, lane);
    bool ok = true;
    for (int j = 0; j < nch && !*abortp; ++j) {
      const int b = j & 1;
      // dA's buffer b was read by dq(j - 2), which completed before dP(j)
      if (!mbar_wait(&dp_full[b], (j >> 1) & 1, WAIT_CYCLES) || !mbar_wait(&gready[j % NG], (j / NG) & 1, WAIT_CYCLES)) {
        ok = false;
        break;
      }
      tc_fence_after();
      decay_mask<false>(tDP(b), lane_off, qw, lane, sm + DAF + b * 8192, nullptr, slot_of(j));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&p_ready[b]);
      mbar_arrive(&gfree[j % NG]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
  } else if (warp < 10) {
    // ---------------- state ----------------
    const int qw = warp & 3, c = qw * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    float Sr[64];
    {
      const float *h0row = a.h0 ? a.h0 + ((d * H + h) * KD + c) * VD : nullptr;
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const float4 x = h0row ? *reinterpret_cast<const float4 *>(h0row + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        Sr[i] = x.x;
        Sr[i + 1] = x.y;
        Sr[i + 2] = x.z;
        Sr[i + 3] = x.w;
      }
    }
    store_state_row(sm + S + 16384, c, Sr);  // S_in of chunk 0
    fence_async_smem();
    mbar_arrive(&s_ready[1]);
    bool ok = true;
    for (int j = 0; j < nch && !*abortp; ++j) {
      const int b = j & 1;
      // S's buffer b was last read by dq(j - 1)
      if (!mbar_wait(&u_full[b], (j >> 1) & 1, WAIT_CYCLES) || !mbar_wait(&gready[j % NG], (j / NG) & 1, WAIT_CYCLES) ||
          (j >= 1 && !mbar_wait(&dq_full[(j - 1) & 1], ((j - 1) >> 1) & 1, WAIT_CYCLES))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float eGam = lds_f1(smem_u32(slot_of(j)) + 4u * G_EGAM);
#pragma unroll
      for (int cp = 0; cp < 64; cp += 32) {
        uint32_t r[32];
        tmem_ld32(tU(b) + lane_off + cp, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) Sr[cp + i] = fmaf(eGam, Sr[cp + i], __uint_as_float(r[i]));
      }
      store_state_row(sm + S + b * 16384, c, Sr);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&s_ready[b]);
      mbar_arrive(&gfree[j % NG]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
    // <dht, S_T> of this (document, head)
    if (a.dht) {  // every state thread takes this branch (named barrier inside)
      const float *drow = a.dht + ((d * H + h) * KD + c) * VD;
      float p = 0.f;
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(drow + i);
        p += Sr[i] * x.x + Sr[i + 1] * x.y + Sr[i + 2] * x.z + Sr[i + 3] * x.w;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
      if (lane == 0) red[qw] = p;
      named_bar(4, 128);
      if (qw == 0 && lane == 0) a.sdht[d * H + h] = red[0] + red[1] + red[2] + red[3];
    }
  } else if (warp < 14) {
    // ---------------- dq_h out, q . dq_h ----------------
    const int qw = warp & 3, rl = lane & 15, row = qw * 16 + rl;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    bool ok = true;
    for (int j = 0; j < nch && !*abortp; ++j) {
      const int b = j & 1, s = j % NS;
      if (!mbar_wait(&dq_full[b], (j >> 1) & 1, WAIT_CYCLES)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int L = chunk_len(j);
      float dot = reduce_warp_rows(tDQ(b), lane_off, qw, lane, L, sm + DQT + qw * 4096, sm + Q + s * 16384,
                                   &maps.dqa, hq, (int)chunk_tok(j));
      tc_fence_before();
      mbar_arrive(&dq_free[b]);
      mbar_arrive(&empty[s]);
      dot += __shfl_xor_sync(0xffffffffu, dot, 16);
      if (lane < 16 && row < L) a.qdq[(chunk_tok(j) + row) * H + h] = dot;
    }
    if (!ok) atomicExch(&abort_flag, 1);
    if (lane == 0) bulk_wait_all();
  } else {
    // ---------------- gate ----------------
    const int tid = (int)threadIdx.x - 448;
    auto load_g = [&](int jj) -> float {
      if (jj >= nch || tid >= chunk_len(jj)) return 0.f;
      return ldg_early(a.g + (chunk_tok(jj) + tid) * H + h);
    };
    float gnext = load_g(0), gnext2 = load_g(1);
    bool ok = true;
    for (int j = 0; j < nch; ++j) {
      // the 64 threads leave together (named barriers in gate_factors)
      if (named_bar_any(2, 64, !ok || *abortp)) break;
      const int gsl = j % NG, b = j & 1, s = j % NS, L = chunk_len(j);
      float *gs = slot_of(j);
      // slot of j - NG read by the mask and state steps; vt / dot buffers by
      // U(j - 2) and dq(j - 2)
      if ((j >= NG && !mbar_wait(&gfree[gsl], ((j / NG) - 1) & 1, WAIT_CYCLES)) ||
          (j >= 2 && (!mbar_wait(&u_full[b], ((j - 2) >> 1) & 1, WAIT_CYCLES) ||
                      !mbar_wait(&dq_full[b], ((j - 2) >> 1) & 1, WAIT_CYCLES))))
        ok = false;
      const float gt = gnext;
      gnext = gnext2;
      gnext2 = load_g(j + 2);
      float egr, eg;
      gate_factors(gs, tid, lane, L, a.scale, gt, 2, egr, eg);
      if (!ok || !mbar_wait(&full[s], (j / NS) & 1, WAIT_CYCLES)) {
        ok = false;
        continue;
      }
      {
        const uint8_t *vs = sm + V + s * 8192, *ds = sm + DO + s * 8192;
        uint8_t *vd = sm + VT + b * 8192, *dd = sm + DOT + b * 8192;
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          const uint32_t off = sw128_off(tid, c, 64);
          const uint4 x = lds_u4(smem_u32(vs) + off);
          st_shared_v4(smem_u32(vd + off), scale_bf16x2(x.x, egr), scale_bf16x2(x.y, egr), scale_bf16x2(x.z, egr),
                       scale_bf16x2(x.w, egr));
          const uint4 y = lds_u4(smem_u32(ds) + off);
          st_shared_v4(smem_u32(dd + off), scale_bf16x2(y.x, eg), scale_bf16x2(y.y, eg), scale_bf16x2(y.z, eg),
                       scale_bf16x2(y.w, eg));
        }
      }
      fence_async_smem();
      mbar_arrive(&gready[gsl]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
  }
#undef SSD_FAIL
  tc_fence_before();
  __syncthreads();
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// =========================================================================
// pass B: chunks in reverse (iteration i takes chunk nch - 1 - i)
//   warp 0       TMA (q, k, v, do; 2 stages)
//   warp 1       MMA: QK = q k^T, dP = do v^T, W = q^T dot,
//                dV1 = A^T do, dV2 = k dS, dK = dA^T q + vt dS^T (QK / dP
//                of the next chunk go before dV / dK of this one)
//   warps 2..5   mask: A = QK (.) F, dA = dP (.) F (bf16)
//   warps 6..9   state: dS (fp32 in registers), bf16 copy, dh0 at the end;
//                then dv of the chunk
//   warps 10..13 dk_h tile -> reduce-add; dg
//   warps 14, 15 gate: the gate slot, vt, dot
// TMEM: QK at 0, dP at 64, W at 128 (M = 128), dV1 at 192, dV2 at 256,
// dK at 320 (64 x 128).
// =========================================================================
__global__ void __launch_bounds__(512, 1) ssd_bwd_b_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using namespace pbs;
  using namespace gsl;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[NS], empty[NS], gready[NG], gfree[NG], pd_full, w_full, dv_full, dk_full, p_ready, ds_ready[2],
      tm_free, drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float wsum[4];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t H = a.H;
  const int h = (int)((int64_t)blockIdx.x % H);
  const int hq = a.hq_div > 1 ? h / a.hq_div : h;
  const int64_t u = a.units.at((int64_t)blockIdx.x / H);
  const Unit un = a.units.get(u);
  const int64_t d = un.doc, s0 = un.start, s1 = un.end;
  const int nch = (int)((s1 - s0 + C - 1) / C);
  // iteration i works on chunk nch - 1 - i
  auto chunk_tok = [&](int i) -> int64_t { return s0 + (int64_t)(nch - 1 - i) * C; };
  auto chunk_len = [&](int i) -> int { return (int)min((int64_t)C, s1 - chunk_tok(i)); };
  auto slot_of = [&](int i) -> float * { return reinterpret_cast<float *>(sm + GS + (i % NG) * GSLOT); };

  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 129);  // the MMA commit and the 128 threads that read k
    }
    for (int i = 0; i < NG; ++i) {
      mbar_init(&gready[i], 64);
      mbar_init(&gfree[i], 384);  // mask, state and output warpgroups
    }
    mbar_init(&pd_full, 1);
    mbar_init(&w_full, 1);
    mbar_init(&dv_full, 1);
    mbar_init(&dk_full, 1);
    mbar_init(&p_ready, 128);
    mbar_init(&ds_ready[0], 128);
    mbar_init(&ds_ready[1], 128);
    mbar_init(&tm_free, 256);  // dv (state warpgroup) and dk (output warpgroup) read out
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base, sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
#define SSD_FAIL                \
  {                             \
    atomicExch(&abort_flag, 1); \
    break;                      \
  }
  const uint32_t tQK = tbase, tDP = tbase + 64, tW = tbase + 128, tV1 = tbase + 192, tV2 = tbase + 256,
                 tDK = tbase + 320;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dout);
      int issued = 0;
      for (int i = 0; i < nch; ++i) {
        const int s = i % NS;
        if (i >= NS && !mbar_wait(&empty[s], ((i / NS) - 1) & 1, WAIT_CYCLES)) SSD_FAIL
        if (*abortp) break;
        const int tok = (int)chunk_tok(i);
        mbar_expect_tx(&full[s], 16384 + 16384 + 8192 + 8192);
        tma_load_3d(sm + Q + s * 16384, &maps.q, 0, hq, tok, &full[s]);
        tma_load_3d(sm + Q + s * 16384 + 8192, &maps.q, 64, hq, tok, &full[s]);
        tma_load_3d(sm + K + s * 16384, &maps.k, 0, hq, tok, &full[s]);
        tma_load_3d(sm + K + s * 16384 + 8192, &maps.k, 64, hq, tok, &full[s]);
        tma_load_3d(sm + V + s * 8192, &maps.v, 0, h, tok, &full[s]);
        tma_load_3d(sm + DO + s * 8192, &maps.dout, 0, h, tok, &full[s]);
        // the tiles of chunk i + 2 into L2 ahead of their load
        if (i + 2 < nch) {
          const int tp = (int)chunk_tok(i + 2);
          tma_prefetch_3d(&maps.q, 0, hq, tp);
          tma_prefetch_3d(&maps.q, 64, hq, tp);
          tma_prefetch_3d(&maps.k, 0, hq, tp);
          tma_prefetch_3d(&maps.k, 64, hq, tp);
          tma_prefetch_3d(&maps.v, 0, h, tp);
          tma_prefetch_3d(&maps.dout, 0, h, tp);
        }
        issued = i + 1;
      }
      for (int i = max(0, issued - NS); i < issued; ++i)
        if (!mbar_wait(&full[i % NS], (i / NS) & 1, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idKK = idesc_bf16(64, 64, false, false);   // q k^T, do v^T
      constexpr uint32_t idW = idesc_bf16(128, 64, true, true);     // q^T dot
      constexpr uint32_t idV1 = idesc_bf16(64, 64, true, true);     // A^T do
      constexpr uint32_t idV2 = idesc_bf16(64, 64, false, true);    // k dS
      constexpr uint32_t idK1 = idesc_bf16(64, 128, true, true);    // dA^T q
      constexpr uint32_t idK2 = idesc_bf16(64, 128, false, false);  // vt dS^T
      // QK, dP of a chunk (their TMEM was read by the mask step of the chunk before)
      auto issue_qkdp = [&](int ii) {
        const int si = ii % NS;
        const uint32_t qa = sbase + Q + si * 16384, ka = sbase + K + si * 16384, va = sbase + V + si * 8192,
                       da = sbase + DO + si * 8192;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tQK, kdesc(qa, ks, 64), kdesc(ka, ks, 64), idKK, ks);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tDP, kdesc(da, ks, 64), kdesc(va, ks, 64), idKK, ks);
        mma_commit(&pd_full);
      };
      if (nch > 0) {
        const bool ok0 = mbar_wait(&full[0], 0, WAIT_CYCLES);
        tc_fence_after();
        if (ok0)
          issue_qkdp(0);
        else
          atomicExch(&abort_flag, 1);
      }
      // Order per chunk i: W(i); then, once the mask step of i has read QK /
      // dP, QK / dP of i + 1 if its tiles have landed (so that the next mask
      // step overlaps dV / dK of i), dV / dK of i, and QK / dP of i + 1 if
      // they were not issued before.
      for (int i = 0; i < nch && !*abortp; ++i) {
        const int s = i % NS, b = i & 1;
        const uint32_t qa = sbase + Q + s * 16384, ka = sbase + K + s * 16384, da = sbase + DO + s * 8192;
        // W = q^T dot; the state step of i - 1 has read W (it wrote dS_i after)
        if (!mbar_wait(&gready[i % NG], (i / NG) & 1, WAIT_CYCLES) ||
            !mbar_wait(&ds_ready[b], (i >> 1) & 1, WAIT_CYCLES))
          SSD_FAIL
        tc_fence_after();
        {
          const uint32_t dot = sbase + DOT + b * 8192;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tW, mdesc(qa, ks, 8192), mdesc(dot, ks, 8192), idW, ks);
          mma_commit(&w_full);
        }
        // A and dA masked (QK / dP read); dV / dK TMEM read out by the steps of i - 1
        if (!mbar_wait(&p_ready, i & 1, WAIT_CYCLES) || (i >= 1 && !mbar_wait(&tm_free, (i - 1) & 1, WAIT_CYCLES)))
          SSD_FAIL
        tc_fence_after();
        // QK / dP of i + 1 first if its tiles are in (never wait for them here:
        // their stage is released by the output step of i - 1)
        bool next_done = i + 1 >= nch;
        if (!next_done && mbar_test_wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1)) {
          tc_fence_after();
          issue_qkdp(i + 1);
          next_done = true;
        }
        {
          const uint32_t Aa = sbase + A, dfa = sbase + DAF, dsa = sbase + DS + b * 16384, vt = sbase + VT + b * 8192;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tV1, mdesc(Aa, ks, 8192), mdesc(da, ks, 8192), idV1, ks);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) mma_bf16(tV2, kdesc(ka, ks, 64), mdesc(dsa, ks, 16384), idV2, ks);
          mma_commit(&dv_full);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tDK, mdesc(dfa, ks, 8192), mdesc(qa, ks, 8192), idK1, ks);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tDK, kdesc(vt, ks, 64), kdesc(dsa, ks, 128), idK2, 1);
          mma_commit(&dk_full);
          mma_commit(&empty[s]);
        }
        if (!next_done) {
          if (!mbar_wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1, WAIT_CYCLES)) SSD_FAIL
          tc_fence_after();
          issue_qkdp(i + 1);
        }
      }
      mma_commit(&drain);
      if (!mbar_wait(&drain, 0, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else if (warp < 6) {
    // ---------------- mask: A = QK (.) F, dA = dP (.) F ----------------
    const int qw = warp & 3;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    mask_tile_init(sm + A, qw, lane);
    mask_tile_init(sm + DAF, qw, lane);
    bool ok = true;
    for (int i = 0; i < nch && !*abortp; ++i) {
      if (!mbar_wait(&pd_full, i & 1, WAIT_CYCLES) || !mbar_wait(&gready[i % NG], (i / NG) & 1, WAIT_CYCLES)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t wa[2][8], wd[2][8];
      decay_tile_regs(tQK, lane_off, qw, lane, slot_of(i), wa);
      decay_tile_regs(tDP, lane_off, qw, lane, slot_of(i), wd);
      // A and dA tiles: read by dV / dK of i - 1, which may still be running
      if (i >= 1 && (!mbar_wait(&dv_full, (i - 1) & 1, WAIT_CYCLES) || !mbar_wait(&dk_full, (i - 1) & 1, WAIT_CYCLES))) {
        ok = false;
        break;
      }
      decay_tile_store(sm + A, qw, lane, wa);
      decay_tile_store(sm + DAF, qw, lane, wd);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&p_ready);
      mbar_arrive(&gfree[i % NG]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
  } else if (warp < 10) {
    // ---------------- state gradient ----------------
    const int qw = warp & 3, c = qw * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    float Dr[64];
    {
      const float *drow = a.dht ? a.dht + ((d * H + h) * KD + c) * VD : nullptr;
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const float4 x = drow ? *reinterpret_cast<const float4 *>(drow + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        Dr[i] = x.x;
        Dr[i + 1] = x.y;
        Dr[i + 2] = x.z;
        Dr[i + 3] = x.w;
      }
    }
    store_state_row(sm + DS, c, Dr);  // the gradient leaving the last chunk
    fence_async_smem();
    mbar_arrive(&ds_ready[0]);
    bool ok = true;
    for (int i = 0; i < nch && !*abortp; ++i) {
      const int nb = (i + 1) & 1;
      // dS's buffer nb was last read by dV / dK of i - 1, which completed
      // before W(i)
      if (!mbar_wait(&w_full, i & 1, WAIT_CYCLES) || !mbar_wait(&gready[i % NG], (i / NG) & 1, WAIT_CYCLES)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float eGam = lds_f1(smem_u32(slot_of(i)) + 4u * G_EGAM);
#pragma unroll
      for (int cp = 0; cp < 64; cp += 32) {
        uint32_t r[32];
        tmem_ld32(tW + lane_off + cp, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int k = 0; k < 32; ++k) Dr[cp + k] = fmaf(eGam, Dr[cp + k], __uint_as_float(r[k]));
      }
      if (i + 1 < nch) {
        store_state_row(sm + DS + nb * 16384, c, Dr);
        fence_async_smem();
      }
      tc_fence_before();
      mbar_arrive(&ds_ready[nb]);
      // dv = A^T do + exp(Gam - G_s) (k dS)_s
      if (!mbar_wait(&dv_full, i & 1, WAIT_CYCLES)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        const int rl = lane & 15, row = qw * 16 + rl, L = chunk_len(i);
        const bool second = lane >= 16;
        const float egr = lds_f1(smem_u32(slot_of(i)) + 4u * (G_EGR + row));
        __nv_bfloat16 *vrow = a.dv + ((chunk_tok(i) + row) * H + h) * VD;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          uint32_t xa[16], xb[16], pa[16], pb[16];
          tmem_ld16(tV1 + lane_off + 16 * k, xa);
          tmem_ld16(tV1 + lane_off + 32 + 16 * k, xb);
          tmem_ld16(tV2 + lane_off + 16 * k, pa);
          tmem_ld16(tV2 + lane_off + 32 + 16 * k, pb);
          tmem_ld_wait(xa);
          tmem_tie(xb);
          tmem_tie(pa);
          tmem_tie(pb);
          float y[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t xs = __shfl_sync(0xffffffffu, xb[e], rl), ps = __shfl_sync(0xffffffffu, pb[e], rl);
            y[e] = fmaf(egr, __uint_as_float(second ? ps : pa[e]), __uint_as_float(second ? xs : xa[e]));
          }
          if (row < L) {
            __nv_bfloat16 *dst = vrow + (second ? 32 : 0) + 16 * k;
            st_global_v4(dst, pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                         pack_bf16(y[6], y[7]));
            st_global_v4(dst + 8, pack_bf16(y[8], y[9]), pack_bf16(y[10], y[11]), pack_bf16(y[12], y[13]),
                         pack_bf16(y[14], y[15]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tm_free);
      mbar_arrive(&gfree[i % NG]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
    if (a.dh0 && !*abortp) {
      float *dst = a.dh0 + ((d * H + h) * KD + c) * VD;
#pragma unroll
      for (int i = 0; i < 64; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(Dr[i], Dr[i + 1], Dr[i + 2], Dr[i + 3]);
    }
  } else if (warp < 14) {
    // ---------------- dk_h, dg ----------------
    const int qw = warp & 3, rl = lane & 15, row = qw * 16 + rl;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    float carry = a.dht ? a.sdht[d * H + h] : 0.f;  // sum over later tokens + <dht, S_T>
    bool ok = true;
    for (int i = 0; i < nch; ++i) {
      // the 128 threads leave together (named barriers below)
      if (named_bar_any(3, 128, !ok || *abortp)) break;
      const int s = i % NS;
      const int L = chunk_len(i);
      const int64_t tok0 = chunk_tok(i);
      // q . dq_h of the row (pass A's result), loaded while dk_h is computed
      const float qdq = row < L ? ldg_early(a.qdq + (tok0 + row) * H + h) : 0.f;
      if (!mbar_wait(&dk_full, i & 1, WAIT_CYCLES)) ok = false;
      tc_fence_after();
      // dk_h leaves TMEM first, so that the next chunk's products need not
      // wait for the reduce
      float y[4][16];
      tmem_rows128(tDK, lane_off, lane, y);
      tc_fence_before();
      mbar_arrive(&tm_free);
      float kdk = reduce_rows(y, qw, lane, L, sm + DKT + qw * 4096, sm + K + s * 16384, &maps.dka, hq, (int)tok0);
      mbar_arrive(&empty[s]);
      // dg: reverse sum over the chunk of q . dq_h - k . dk_h, plus the carry
      kdk += __shfl_xor_sync(0xffffffffu, kdk, 16);
      float x = (row < L) ? qdq - kdk : 0.f;
      // suffix sum over the warp's 16 rows (lanes 0..15; lanes 16..31 mirror them)
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, x, o, 16);
        if (rl + o < 16) x += y;
      }
      if (lane == 0) wsum[qw] = x;  // the warp's total (row 16 qw)
      named_bar(3, 128);
      float later = carry;
#pragma unroll
      for (int w = 0; w < 4; ++w)
        if (w > qw) later += wsum[w];
      if (lane < 16 && row < L) a.dg[(tok0 + row) * H + h] = later + x;
      carry += wsum[0] + wsum[1] + wsum[2] + wsum[3];
      named_bar(3, 128);
      mbar_arrive(&gfree[i % NG]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
    if (lane == 0) bulk_wait_all();
  } else {
    // ---------------- gate ----------------
    const int tid = (int)threadIdx.x - 448;
    auto load_g = [&](int ii) -> float {
      if (ii >= nch || tid >= chunk_len(ii)) return 0.f;
      return ldg_early(a.g + (chunk_tok(ii) + tid) * H + h);
    };
    float gnext = load_g(0), gnext2 = load_g(1);
    bool ok = true;
    for (int i = 0; i < nch; ++i) {
      // the 64 threads leave together (named barriers in gate_factors)
      if (named_bar_any(2, 64, !ok || *abortp)) break;
      const int gsl = i % NG, b = i & 1, s = i % NS, L = chunk_len(i);
      float *gs = slot_of(i);
      // slot of i - NG read by the mask, state and output steps; vt / dot
      // buffers by dK(i - 2) and W(i - 2), both complete before W(i - 1)
      if ((i >= NG && !mbar_wait(&gfree[gsl], ((i / NG) - 1) & 1, WAIT_CYCLES)) ||
          (i >= 2 && !mbar_wait(&w_full, (i - 1) & 1, WAIT_CYCLES)))
        ok = false;
      const float gt = gnext;
      gnext = gnext2;
      gnext2 = load_g(i + 2);
      float egr, eg;
      gate_factors(gs, tid, lane, L, a.scale, gt, 2, egr, eg);
      if (!ok || !mbar_wait(&full[s], (i / NS) & 1, WAIT_CYCLES)) {
        ok = false;
        continue;
      }
      {
        const uint8_t *vs = sm + V + s * 8192, *ds = sm + DO + s * 8192;
        uint8_t *vd = sm + VT + b * 8192, *dd = sm + DOT + b * 8192;
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          const uint32_t off = sw128_off(tid, c, 64);
          const uint4 x = lds_u4(smem_u32(vs) + off);
          st_shared_v4(smem_u32(vd + off), scale_bf16x2(x.x, egr), scale_bf16x2(x.y, egr), scale_bf16x2(x.z, egr),
                       scale_bf16x2(x.w, egr));
          const uint4 y = lds_u4(smem_u32(ds) + off);
          st_shared_v4(smem_u32(dd + off), scale_bf16x2(y.x, eg), scale_bf16x2(y.y, eg), scale_bf16x2(y.z, eg),
                       scale_bf16x2(y.w, eg));
        }
      }
      fence_async_smem();
      mbar_arrive(&gready[gsl]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
  }
#undef SSD_FAIL
  tc_fence_before();
  __syncthreads();
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// fp32 group accumulators -> bf16 gradients (n elements, multiple of 4)
__global__ void ssd_round_grads_kernel(const float4 *__restrict__ dqa, const float4 *__restrict__ dka,
                                       uint2 *__restrict__ dq, uint2 *__restrict__ dk, int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    const float4 x = dqa[i], y = dka[i];
    dq[i] = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
    dk[i] = make_uint2(pack_bf16(y.x, y.y), pack_bf16(y.z, y.w));
  }
}

// ---- host ----------------------------------------------------------------

struct BwdLayout {
  size_t off_order, off_dqa, off_dka, off_qdq, off_sdht, total;
};
static size_t al256b(size_t x) { return (x + 255) & ~(size_t)255; }
static BwdLayout bwd_layout(const glacore_problem *p) {
  BwdLayout L;
  const size_t BT = (size_t)(p->B * p->T), acc = BT * (size_t)p->Hqk * KD * sizeof(float);
  size_t off = 0;
  L.off_order = off;
  if (p->segment_ids) off = al256b(off + (size_t)p->n_seqs * sizeof(int32_t));
  L.off_dqa = off;
  off = al256b(off + acc);
  L.off_dka = off;
  off = al256b(off + acc);
  L.off_qdq = off;
  off = al256b(off + BT * (size_t)p->H * sizeof(float));
  L.off_sdht = off;
  off = al256b(off + (size_t)p->n_seqs * (size_t)p->H * sizeof(float));
  L.total = off;
  return L;
}

size_t bwd_workspace_bytes(const glacore_problem *p) { return bwd_layout(p).total; }

cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO, const float *dht,
                void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws, cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
  if (const cudaError_t be = bind_context()) return be;
  const BwdLayout Lo = bwd_layout(p);
  float *dqa = (float *)(ws + Lo.off_dqa), *dka = (float *)(ws + Lo.off_dka);
  BwdMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (!make_map(&maps.q, pr.q, true, KD, pr.Hqk, pr.BT, 64, pr.qs) ||
      !make_map(&maps.k, pr.k, true, KD, pr.Hqk, pr.BT, 64, pr.ks) ||
      !make_map(&maps.v, pr.v, true, VD, pr.H, pr.BT, 64, pr.vs) ||
      !make_map(&maps.dout, dO, true, VD, pr.H, pr.BT, 64) ||
      !make_map(&maps.dqa, dqa, false, KD, pr.Hqk, pr.BT, 32, 0, 16) ||
      !make_map(&maps.dka, dka, false, KD, pr.Hqk, pr.BT, 32, 0, 16))
    return cudaErrorInvalidValue;
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.units.docs = docs;
  a.units.order = docs.start ? (const int32_t *)(ws + Lo.off_order) : nullptr;
  a.H = pr.H;
  a.hq_div = (int32_t)(pr.H / pr.Hqk);
  a.scale = pr.scale;
  a.g = pr.g;
  a.h0 = pr.h0;
  a.dht = dht;
  a.dh0 = dh0;
  a.dv = (__nv_bfloat16 *)dv;
  a.dg = dg;
  a.qdq = (float *)(ws + Lo.off_qdq);
  a.sdht = (float *)(ws + Lo.off_sdht);
  a.err = pr.err;
  cudaError_t e;
  const size_t acc = (size_t)pr.BT * pr.Hqk * KD * sizeof(float);
  if ((e = cudaMemsetAsync(dqa, 0, acc, st)) != cudaSuccess || (e = cudaMemsetAsync(dka, 0, acc, st)) != cudaSuccess)
    return e;
  if (a.units.order &&
      (e = launch_order_units(a.units, docs.n, (int32_t *)(ws + Lo.off_order), st)) != cudaSuccess)
    return e;
  const int smem_a = pas::BYTES + 1024, smem_b = pbs::BYTES + 1024;
  if ((e = cudaFuncSetAttribute(ssd_bwd_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_a)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(ssd_bwd_b_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_b)) != cudaSuccess)
    return e;
  const unsigned grid = (unsigned)(docs.n * pr.H);
  ssd_bwd_a_kernel<<<grid, 512, smem_a, st>>>(maps, a);
  mark_launch("ssd_bwd_a_kernel", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  ssd_bwd_b_kernel<<<grid, 512, smem_b, st>>>(maps, a);
  mark_launch("ssd_bwd_b_kernel", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t n4 = pr.BT * pr.Hqk * KD / 4;
  ssd_round_grads_kernel<<<(unsigned)std::min<int64_t>((n4 + 255) / 256, 152 * 8), 256, 0, st>>>(
      (const float4 *)dqa, (const float4 *)dka, (uint2 *)dq, (uint2 *)dk, n4);
  mark_launch("ssd_round_grads", st);
  return cudaGetLastError();
}

}  // namespace ssd
}  // namespace glacore
