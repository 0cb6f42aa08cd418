// tc_gla_bwd.cu -- tcgen05 backward of GLA (bf16, K = V = 128, C = 64).
//
// FLAT blog (trainstation-project.github.io/blog/flat), "Backward
// Recurrence" and "Backward Kernels": the state gradient runs backwards in
// time; per chunk the input gradients read off the carried state (dq) and
// the carried state gradient (dk, dv); the gate gradient is the suffix sum
// of q (.) dq - k (.) dk.  States are recomputed here, not stored by the
// forward.  Two kernels:
//
//  pass A (chunks in order, state S recomputed on chip, fp32 in TMEM):
//     dP  = (dO V^T) masked to s <= t
//     dq  = scale exp(G) (dO S_prev^T + dP kt)      kt = k exp(-G)
//     dgp_t = sum_{r >= t in chunk} q_r dq_r        (fp32 scratch)
//     S  <- diag(exp(Gam)) (S + kt^T V)
//     bvec = (S_T (.) dht) 1_V                      (final-state term of dg)
//  pass B (chunks in reverse, dH fp32 in TMEM):
//     dHh = diag(exp(Gam)) dH
//     dk  = exp(-G) (dP^T qt + V dHh^T)             qt = scale q exp(G)
//     dv  = P^T dO + kt dHh                          P = (qt kt^T) masked
//     dg_t = dgp_t - sum_{r >= t in chunk} k_r dk_r + carry,
//     carry <- carry + (chunk totals)               (starts at bvec)
//     dH <- dHh + qt^T dO;  dh0 = dH at the document start
//
// dq, dk, dv are produced transposed (rows = key channel or value column)
// as M = 128 tcgen05 accumulators, so thread c of the epilogue warpgroup
// reads row c of TMEM and owns channel c for the suffix sums.  Thread roles
// as in the forward: warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..9 prep
// (thread = one key channel x 32 tokens; it stages exp(+-G) into its own
// TMEM lane), warps 10..13 epilogue.
#include "tc_common.cuh"

namespace glacore {
namespace tc {

struct BwdMaps {
  CUtensorMap q, k, v, dO;
};
struct BwdArgs {
  Docs docs;
  int64_t H;
  float scale;
  const float *g;
  const float *h0;
  const float *dht;
  __nv_bfloat16 *dq, *dk, *dv;
  float *dg, *dh0;
  float *dgp;   // scratch [BT, H, K] fp32
  float *bvec;  // scratch [n_docs, H, K] fp32
  int *err;
};

#define BW_FAIL_AND_BREAK         \
  {                               \
    atomicExch(&abort_flag, 1);   \
    break;                        \
  }

// Gate work of one chunk for a per-channel prep thread (channel c, tokens
// 32 th .. 32 th + 31): loads its 32 gates, exchanges the half-chunk
// product of exp(g) with the other half (xch, named barrier 1 over the 256
// prep threads) and returns exp(g) per token plus the products needed for
// exp(G_t) (prefix) and exp(Gam - G_t) (suffix).  Tokens t >= L get g = 0.
struct ChanGate {
  float x[32];
  float before;  // product of exp(g) over the tokens before this half
  float after;   // product over the tokens after this half
  float total;   // exp(Gam)
};
__device__ __forceinline__ void load_gates(ChanGate &cg, const float *g, int64_t tok0, int64_t H,
                                           int h, int c, int th, int L) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int t = 32 * th + i;
    cg.x[i] = t < L ? __ldg(g + ((tok0 + t) * H + h) * KD + c) : 0.f;
  }
}
__device__ __forceinline__ void exchange_gates(ChanGate &cg, float *xch, int c, int th, int L) {
  float p = 1.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    cg.x[i] = (32 * th + i < L) ? __expf(cg.x[i]) : 1.f;
    p *= cg.x[i];
  }
  xch[th * 128 + c] = p;
  named_bar(1, 256);
  const float o = xch[(1 - th) * 128 + c];
  cg.before = th ? o : 1.f;
  cg.after = th ? 1.f : o;
  cg.total = p * o;
}

// ===========================================================================
// pass A
// ===========================================================================
namespace asm_ {  // shared-memory carve-up (bytes)
constexpr int NS = 2;
constexpr uint32_t Q = 0;          // 2 x 16 KB raw q
constexpr uint32_t K = 32768;      // 2 x 16 KB k, then kt in place
constexpr uint32_t V = 65536;      // 2 x 16 KB
constexpr uint32_t DO = 98304;     // 2 x 16 KB
constexpr uint32_t DP = 131072;    // 2 x 8 KB masked dP (bf16 [t][s])
constexpr uint32_t S = 147456;     // 2 x 32 KB S (bf16 [c][v], K-major A)
constexpr uint32_t XCH = 212992;   // 2 x 2 x 128 fp32
constexpr uint32_t BYTES = 215040;
}  // namespace asm_

__global__ void __launch_bounds__(448)
    gla_bwd_dq_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[asm_::NS], empty[asm_::NS], prep_done[asm_::NS], dp_full[2],
      dp_ready[2], dq_full[2], u_full, s_ready, eg_ready[2], eg_free[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int64_t d = blockIdx.x;
  const int64_t H = a.H;
  int64_t s0, s1;
  a.docs.range(d, s0, s1);
  const int nch = (int)((s1 - s0 + C - 1) / C);

  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < asm_::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + 128);  // MMA commit + epilogue (reads raw q)
      mbar_init(&prep_done[i], 256);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&dp_full[i], 1);
      mbar_init(&dp_ready[i], 128);
      mbar_init(&dq_full[i], 1);
      mbar_init(&eg_ready[i], 256);
      mbar_init(&eg_free[i], 128);
    }
    mbar_init(&u_full, 1);
    mbar_init(&s_ready, 128);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
  // TMEM columns
  const uint32_t tDP = tbase, tDQ = tbase + 128, tS = tbase + 256, tEG = tbase + 384;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dO);
      for (int j = 0; j < nch; ++j) {
        const int st = j % asm_::NS;
        if (j >= asm_::NS && !mbar_wait(&empty[st], ((j / asm_::NS) - 1) & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)(s0 + (int64_t)j * C);
        if (j + 2 < nch) {
          const int tp = tok + 2 * C;
          for (int x = 0; x < 128; x += 64) {
            tma_prefetch_3d(&maps.q, x, h, tp);
            tma_prefetch_3d(&maps.k, x, h, tp);
            tma_prefetch_3d(&maps.v, x, h, tp);
            tma_prefetch_3d(&maps.dO, x, h, tp);
          }
        }
        mbar_expect_tx(&full[st], 4 * 16384);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(sm + asm_::Q + st * 16384 + x * 8192, &maps.q, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + asm_::K + st * 16384 + x * 8192, &maps.k, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + asm_::V + st * 16384 + x * 8192, &maps.v, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + asm_::DO + st * 16384 + x * 8192, &maps.dO, 64 * x, h, tok, &full[st]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idDP = idesc_bf16(64, 64, false, false);
      constexpr uint32_t idU = idesc_bf16(128, 128, true, true);
      constexpr uint32_t idQ1 = idesc_bf16(128, 64, false, false);
      constexpr uint32_t idQ2 = idesc_bf16(128, 64, true, false);
      uint32_t ph_prep = 0, ph_dpr = 0;
      for (int j = 0; j < nch; ++j) {
        const int st = j % asm_::NS, b = j & 1;
        const uint32_t qa = sbase + asm_::Q + st * 16384;
        const uint32_t ka = sbase + asm_::K + st * 16384, va = sbase + asm_::V + st * 16384;
        const uint32_t doa = sbase + asm_::DO + st * 16384, dpa = sbase + asm_::DP + b * 8192;
        const uint32_t Sa = sbase + asm_::S + (b ^ 1) * 32768;
        (void)qa;
        if (!mbar_wait(&prep_done[st], (ph_prep >> st) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph_prep ^= 1u << st;
        tc_fence_after();
        // dP = dO V^T
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tDP + 64 * b, kdesc(doa, ks, 64), kdesc(va, ks, 64), idDP, ks);
        mma_commit(&dp_full[b]);
        // S (TMEM, = S_prev) += kt^T V
        if (!mbar_wait(&s_ready, j & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tS, mdesc(ka, ks, 8192), mdesc(va, ks, 8192), idU, 1);
        mma_commit(&u_full);
        // dq^T = S_prev dO^T + kt^T dP^T
        if (!mbar_wait(&dp_ready[b], (ph_dpr >> b) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph_dpr ^= 1u << b;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tDQ + 64 * b, kdesc(Sa, ks, 128), kdesc(doa, ks, 64), idQ1, ks);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tDQ + 64 * b, mdesc(ka, ks, 8192), kdesc(dpa, ks, 64), idQ2, 1);
        mma_commit(&dq_full[b]);
        mma_commit(&empty[st]);
      }
    }
  } else if (warp < 10) {
    // ---------------- prep: thread = key channel c, 32 tokens ----------------
    const int qw = warp & 3, th = (warp - 2) >> 2;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    uint32_t ph_full = 0, ph_free = 0;
    for (int j = 0; j < nch; ++j) {
      const int st = j % asm_::NS, b = j & 1;
      const int64_t tok0 = s0 + (int64_t)j * C;
      const int L = (int)min((int64_t)C, s1 - tok0);
      ChanGate cg;
      load_gates(cg, a.g, tok0, H, h, c, th, L);
      if (!mbar_wait(&full[st], (ph_full >> st) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      ph_full ^= 1u << st;
      exchange_gates(cg, reinterpret_cast<float *>(sm + asm_::XCH) + b * 256, c, th, L);
      // exp(G_t) -> TMEM (epilogue scales dq with it); column 63 = exp(Gam)
      if (j >= 2) {
        if (!mbar_wait(&eg_free[b], (ph_free >> b) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph_free ^= 1u << b;
      }
      tc_fence_after();
      {
        uint32_t r[32];
        float pre = cg.before;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          pre *= cg.x[i];
          r[i] = __float_as_uint(pre);
        }
        tmem_st32(tEG + 64 * b + lane_off + 32 * th, r);
      }
      // kt = k exp(-Gam) exp(Gam - G) in place
      {
        const float inv = __frcp_rn(cg.total);
        uint8_t *kt = sm + asm_::K + st * 16384;
        float suf = cg.after;
#pragma unroll
        for (int i = 31; i >= 0; --i) {
          const int t = 32 * th + i;
          const uint32_t ad = smem_u32(kt + sw128_off(t, c, 64));
          const float kv = bf16_bits_to_f32(lds_u16(ad));
          sts_u16(ad, f32_to_bf16_bits(t < L ? kv * suf * inv : 0.f));
          suf *= cg.x[i];
        }
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&prep_done[st]);
      mbar_arrive(&eg_ready[b]);
    }
  } else {
    // ---------------- epilogue: thread = key channel c ----------------
    const int qw = warp & 3;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    // S (TMEM) = h0, bf16 copy for chunk 0's readout
    {
      const float *h0 = a.h0 ? a.h0 + ((d * H + h) * KD + c) * VD : nullptr;
      uint8_t *St = sm + asm_::S + 32768;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(h0 ? h0[32 * cb + i] : 0.f);
        tmem_st32(tS + lane_off + 32 * cb, r);
#pragma unroll
        for (int n = 0; n < 32; n += 8)
          st_shared_v4(smem_u32(St + sw128_off(c, 32 * cb + n, 128)),
                       pack_bf16(__uint_as_float(r[n]), __uint_as_float(r[n + 1])),
                       pack_bf16(__uint_as_float(r[n + 2]), __uint_as_float(r[n + 3])),
                       pack_bf16(__uint_as_float(r[n + 4]), __uint_as_float(r[n + 5])),
                       pack_bf16(__uint_as_float(r[n + 6]), __uint_as_float(r[n + 7])));
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&s_ready);
    }
    uint32_t ph_dpf = 0, ph_dqf = 0, ph_egr = 0;
    // dq epilogue of chunk jj (buffer bb): dq = scale exp(G) acc, suffix of q dq
    auto dq_epilogue = [&](int jj) -> bool {
      const int bb = jj & 1, stt = jj % asm_::NS;
      const int64_t tok0 = s0 + (int64_t)jj * C;
      const int L = (int)min((int64_t)C, s1 - tok0);
      if (!mbar_wait(&dq_full[bb], (ph_dqf >> bb) & 1, WAIT_CYCLES)) return false;
      ph_dqf ^= 1u << bb;
      tc_fence_after();
      const uint8_t *qt = sm + asm_::Q + stt * 16384;
      float suf = 0.f;
#pragma unroll
      for (int half = 1; half >= 0; --half) {
        uint32_t acc[32], eg[32];
        tmem_ld32(tDQ + 64 * bb + lane_off + 32 * half, acc);
        tmem_ld_wait32(acc);
        tmem_ld32(tEG + 64 * bb + lane_off + 32 * half, eg);
        tmem_ld_wait32(eg);
#pragma unroll
        for (int i = 31; i >= 0; --i) {
          const int t = 32 * half + i;
          if (t < L) {
            const float dq = a.scale * __uint_as_float(eg[i]) * __uint_as_float(acc[i]);
            const float qv = bf16_bits_to_f32(lds_u16(smem_u32(qt + sw128_off(t, c, 64))));
            suf += qv * dq;
            const int64_t off = ((tok0 + t) * H + h) * KD + c;
            a.dq[off] = __float2bfloat16_rn(dq);
            a.dgp[off] = suf;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&eg_free[bb]);
      mbar_arrive(&empty[stt]);
      return true;
    };
    bool ok = true;
    for (int j = 0; j < nch && ok; ++j) {
      const int b = j & 1;
      // (1) masked dP -> bf16 operand
      if (!mbar_wait(&dp_full[b], (ph_dpf >> b) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      ph_dpf ^= 1u << b;
      tc_fence_after();
      mask_tile_to_smem(tDP + 64 * b, lane_off, qw, lane, sm + asm_::DP + b * 8192);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&dp_ready[b]);
      // (2) dq of the previous chunk
      if (j >= 1 && !dq_epilogue(j - 1)) BW_FAIL_AND_BREAK
      // (3) S <- exp(Gam) (S_prev + kt^T V): TMEM in place, bf16 copy
      if (!mbar_wait(&u_full, j & 1, WAIT_CYCLES) ||
          !mbar_wait(&eg_ready[b], (ph_egr >> b) & 1, WAIT_CYCLES))
        BW_FAIL_AND_BREAK
      ph_egr ^= 1u << b;
      tc_fence_after();
      {
        uint32_t e1[16];
        tmem_ld16(tEG + 64 * b + lane_off + 48, e1);
        tmem_ld_wait(e1);
        const float eGam = __uint_as_float(e1[15]);
        uint8_t *St = sm + asm_::S + b * 32768;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tS + lane_off + 32 * cb, r);
          tmem_ld_wait32(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(eGam * __uint_as_float(r[i]));
          tmem_st32(tS + lane_off + 32 * cb, r);
#pragma unroll
          for (int n = 0; n < 32; n += 8)
            st_shared_v4(smem_u32(St + sw128_off(c, 32 * cb + n, 128)),
                         pack_bf16(__uint_as_float(r[n]), __uint_as_float(r[n + 1])),
                         pack_bf16(__uint_as_float(r[n + 2]), __uint_as_float(r[n + 3])),
                         pack_bf16(__uint_as_float(r[n + 4]), __uint_as_float(r[n + 5])),
                         pack_bf16(__uint_as_float(r[n + 6]), __uint_as_float(r[n + 7])));
        }
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&s_ready);
    }
    if (!*abortp && nch > 0) {
      if (!dq_epilogue(nch - 1)) atomicExch(&abort_flag, 1);
    }
    // final-state term of the gate gradient: bvec = (S_T (.) dht) 1_V
    if (!*abortp && a.bvec) {
      float acc = 0.f;
      if (a.dht) {
        const float *dh = a.dht + ((d * H + h) * KD + c) * VD;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tS + lane_off + 32 * cb, r);
          tmem_ld_wait32(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc += __uint_as_float(r[i]) * dh[32 * cb + i];
        }
      }
      a.bvec[(d * H + h) * KD + c] = acc;
    }
    (void)ok;
  }
  tc_fence_before();
  __syncthreads();
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ===========================================================================
// pass B
// ===========================================================================
namespace bsm {  // shared-memory carve-up (bytes)
constexpr int NS = 2;
constexpr uint32_t Q = 0;          // 2 x 16 KB q, then qt in place
constexpr uint32_t K = 32768;      // 2 x 16 KB raw k
constexpr uint32_t KT = 65536;     // 2 x 16 KB kt
constexpr uint32_t V = 98304;      // 2 x 16 KB
constexpr uint32_t DO = 131072;    // 2 x 16 KB
constexpr uint32_t P = 163840;     // 8 KB masked P  (bf16 [t][s])
constexpr uint32_t DP = 172032;    // 8 KB masked dP (bf16 [t][s])
constexpr uint32_t DH = 180224;    // 32 KB dHh (bf16 [c][v])
constexpr uint32_t XCH = 212992;   // 2 x 2 x 128 fp32
constexpr uint32_t BYTES = 215040;
}  // namespace bsm

__global__ void __launch_bounds__(448)
    gla_bwd_rev_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[bsm::NS], empty[bsm::NS], prep_done[bsm::NS], pdp_full, pdp_ready,
      dh_ready, kv_full, eg_ready[2], eg_free[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int64_t d = blockIdx.x;
  const int64_t H = a.H;
  int64_t s0, s1;
  a.docs.range(d, s0, s1);
  const int nch = (int)((s1 - s0 + C - 1) / C);

  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < bsm::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1 + 128);  // MMA commit + epilogue (reads raw k)
      mbar_init(&prep_done[i], 256);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&eg_ready[i], 256);
      mbar_init(&eg_free[i], 128);
    }
    mbar_init(&pdp_full, 1);
    mbar_init(&pdp_ready, 128);
    mbar_init(&dh_ready, 128);
    mbar_init(&kv_full, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
  const uint32_t tDH = tbase, tP = tbase + 128, tDP = tbase + 192, tDK = tbase + 256,
                 tDV = tbase + 320, tEG = tbase + 384;

  // chunks are visited in reverse: iteration i handles chunk j = nch - 1 - i
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dO);
      for (int i = 0; i < nch; ++i) {
        const int j = nch - 1 - i, st = i % bsm::NS;
        if (i >= bsm::NS && !mbar_wait(&empty[st], ((i / bsm::NS) - 1) & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)(s0 + (int64_t)j * C);
        if (j - 2 >= 0) {
          const int tp = tok - 2 * C;
          for (int x = 0; x < 128; x += 64) {
            tma_prefetch_3d(&maps.q, x, h, tp);
            tma_prefetch_3d(&maps.k, x, h, tp);
            tma_prefetch_3d(&maps.v, x, h, tp);
            tma_prefetch_3d(&maps.dO, x, h, tp);
          }
        }
        mbar_expect_tx(&full[st], 4 * 16384);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(sm + bsm::Q + st * 16384 + x * 8192, &maps.q, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + bsm::K + st * 16384 + x * 8192, &maps.k, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + bsm::V + st * 16384 + x * 8192, &maps.v, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + bsm::DO + st * 16384 + x * 8192, &maps.dO, 64 * x, h, tok, &full[st]);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idCC = idesc_bf16(64, 64, false, false);
      constexpr uint32_t idMM = idesc_bf16(128, 64, true, true);   // MN-major A and B
      constexpr uint32_t idKK = idesc_bf16(128, 64, false, false); // K-major A and B
      constexpr uint32_t idMK = idesc_bf16(128, 64, true, false);  // MN-major A, K-major B
      constexpr uint32_t idH = idesc_bf16(128, 128, true, true);
      uint32_t ph_prep = 0;
      const uint32_t pa = sbase + bsm::P, dpa = sbase + bsm::DP, dha = sbase + bsm::DH;
      for (int i = 0; i < nch; ++i) {
        const int st = i % bsm::NS;
        const uint32_t qa = sbase + bsm::Q + st * 16384, kta = sbase + bsm::KT + st * 16384;
        const uint32_t va = sbase + bsm::V + st * 16384, doa = sbase + bsm::DO + st * 16384;
        if (!mbar_wait(&prep_done[st], (ph_prep >> st) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph_prep ^= 1u << st;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tP, kdesc(qa, ks, 64), kdesc(kta, ks, 64), idCC, ks);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tDP, kdesc(doa, ks, 64), kdesc(va, ks, 64), idCC, ks);
        mma_commit(&pdp_full);
        if (!mbar_wait(&pdp_ready, i & 1, WAIT_CYCLES) || !mbar_wait(&dh_ready, i & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        tc_fence_after();
        // dk^T = qt^T dP + dHh V^T
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tDK, mdesc(qa, ks, 8192), mdesc(dpa, ks, 8192), idMM, ks);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tDK, kdesc(dha, ks, 128), kdesc(va, ks, 64), idKK, 1);
        // dv^T = dO^T P + dHh^T kt^T
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tDV, mdesc(doa, ks, 8192), mdesc(pa, ks, 8192), idMM, ks);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tDV, mdesc(dha, ks, 16384), kdesc(kta, ks, 64), idMK, 1);
        // dH (= dHh in TMEM) += qt^T dO
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tDH, mdesc(qa, ks, 8192), mdesc(doa, ks, 8192), idH, 1);
        mma_commit(&kv_full);
        mma_commit(&empty[st]);
      }
    }
  } else if (warp < 10) {
    // ---------------- prep: thread = key channel c, 32 tokens ----------------
    const int qw = warp & 3, th = (warp - 2) >> 2;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    uint32_t ph_full = 0, ph_free = 0;
    for (int i = 0; i < nch; ++i) {
      const int j = nch - 1 - i, st = i % bsm::NS, b = i & 1;
      const int64_t tok0 = s0 + (int64_t)j * C;
      const int L = (int)min((int64_t)C, s1 - tok0);
      ChanGate cg;
      load_gates(cg, a.g, tok0, H, h, c, th, L);
      if (!mbar_wait(&full[st], (ph_full >> st) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      ph_full ^= 1u << st;
      exchange_gates(cg, reinterpret_cast<float *>(sm + bsm::XCH) + b * 256, c, th, L);
      const float inv = __frcp_rn(cg.total);
      // qt = scale q exp(G) in place
      {
        uint8_t *q = sm + bsm::Q + st * 16384;
        float pre = cg.before;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int t = 32 * th + u;
          pre *= cg.x[u];
          const uint32_t ad = smem_u32(q + sw128_off(t, c, 64));
          const float qv = bf16_bits_to_f32(lds_u16(ad));
          sts_u16(ad, f32_to_bf16_bits(t < L ? a.scale * qv * pre : 0.f));
        }
      }
      // kt = k exp(-G) (separate tile; raw k is kept for k (.) dk); exp(-G) -> TMEM
      if (i >= 2) {
        if (!mbar_wait(&eg_free[b], (ph_free >> b) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph_free ^= 1u << b;
      }
      tc_fence_after();
      {
        const uint8_t *k = sm + bsm::K + st * 16384;
        uint8_t *kt = sm + bsm::KT + st * 16384;
        uint32_t r[32];
        float suf = cg.after;
#pragma unroll
        for (int u = 31; u >= 0; --u) {
          const int t = 32 * th + u;
          const float e = suf * inv;  // exp(-G_t)
          r[u] = __float_as_uint(e);
          const uint32_t off = sw128_off(t, c, 64);
          const float kv = bf16_bits_to_f32(lds_u16(smem_u32(k + off)));
          sts_u16(smem_u32(kt + off), f32_to_bf16_bits(t < L ? kv * e : 0.f));
          suf *= cg.x[u];
        }
        tmem_st32(tEG + 64 * b + lane_off + 32 * th, r);
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&prep_done[st]);
      mbar_arrive(&eg_ready[b]);
    }
  } else {
    // ---------------- epilogue: thread = key channel / value column c ----------------
    const int qw = warp & 3;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    // dH = dht (or 0)
    {
      const float *dh = a.dht ? a.dht + ((d * H + h) * KD + c) * VD : nullptr;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(dh ? dh[32 * cb + u] : 0.f);
        tmem_st32(tDH + lane_off + 32 * cb, r);
      }
      tmem_st_wait();
    }
    float carry = a.bvec ? a.bvec[(d * H + h) * KD + c] : 0.f;
    uint32_t ph_egr = 0;
    for (int i = 0; i < nch; ++i) {
      const int j = nch - 1 - i, st = i % bsm::NS, b = i & 1;
      const int64_t tok0 = s0 + (int64_t)j * C;
      const int L = (int)min((int64_t)C, s1 - tok0);
      // (1) masked P and dP -> bf16 operands
      if (!mbar_wait(&pdp_full, i & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      tc_fence_after();
      mask_tile_to_smem(tP, lane_off, qw, lane, sm + bsm::P);
      mask_tile_to_smem(tDP, lane_off, qw, lane, sm + bsm::DP);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&pdp_ready);
      // (2) dHh = exp(Gam) dH in TMEM, bf16 copy
      if (!mbar_wait(&eg_ready[b], (ph_egr >> b) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      ph_egr ^= 1u << b;
      tc_fence_after();
      {
        uint32_t e1[16];
        tmem_ld16(tEG + 64 * b + lane_off + 48, e1);
        tmem_ld_wait(e1);
        const float eGam = __frcp_rn(__uint_as_float(e1[15]));  // 1 / exp(-Gam)
        uint8_t *Dt = sm + bsm::DH;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tDH + lane_off + 32 * cb, r);
          tmem_ld_wait32(r);
#pragma unroll
          for (int u = 0; u < 32; ++u) r[u] = __float_as_uint(eGam * __uint_as_float(r[u]));
          tmem_st32(tDH + lane_off + 32 * cb, r);
#pragma unroll
          for (int n = 0; n < 32; n += 8)
            st_shared_v4(smem_u32(Dt + sw128_off(c, 32 * cb + n, 128)),
                         pack_bf16(__uint_as_float(r[n]), __uint_as_float(r[n + 1])),
                         pack_bf16(__uint_as_float(r[n + 2]), __uint_as_float(r[n + 3])),
                         pack_bf16(__uint_as_float(r[n + 4]), __uint_as_float(r[n + 5])),
                         pack_bf16(__uint_as_float(r[n + 6]), __uint_as_float(r[n + 7])));
        }
        tmem_st_wait();
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&dh_ready);
      // (3) dk, dg (thread = channel c) and dv (thread = value column c)
      if (!mbar_wait(&kv_full, i & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      tc_fence_after();
      {
        const uint8_t *k = sm + bsm::K + st * 16384;
        float sk = 0.f, qtot = 0.f;
#pragma unroll
        for (int half = 1; half >= 0; --half) {
          uint32_t acc[32], eg[32];
          tmem_ld32(tDK + lane_off + 32 * half, acc);
          tmem_ld_wait32(acc);
          tmem_ld32(tEG + 64 * b + lane_off + 32 * half, eg);
          tmem_ld_wait32(eg);
#pragma unroll
          for (int u = 31; u >= 0; --u) {
            const int t = 32 * half + u;
            if (t < L) {
              const float dk = __uint_as_float(eg[u]) * __uint_as_float(acc[u]);
              const float kv = bf16_bits_to_f32(lds_u16(smem_u32(k + sw128_off(t, c, 64))));
              sk += kv * dk;
              const int64_t off = ((tok0 + t) * H + h) * KD + c;
              const float qpart = a.dgp[off];
              if (t == 0) qtot = qpart;
              a.dk[off] = __float2bfloat16_rn(dk);
              a.dg[off] = qpart - sk + carry;
            }
          }
        }
        carry += qtot - sk;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t acc[32];
          tmem_ld32(tDV + lane_off + 32 * half, acc);
          tmem_ld_wait32(acc);
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const int t = 32 * half + u;
            if (t < L) a.dv[((tok0 + t) * H + h) * VD + c] = __float2bfloat16_rn(__uint_as_float(acc[u]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&eg_free[b]);
      mbar_arrive(&empty[st]);
    }
    if (!*abortp && a.dh0) {
      float *dst = a.dh0 + ((d * H + h) * KD + c) * VD;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tDH + lane_off + 32 * cb, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int u = 0; u < 32; u += 4)
          *reinterpret_cast<float4 *>(dst + 32 * cb + u) =
              make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]), __uint_as_float(r[u + 2]),
                          __uint_as_float(r[u + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (warp == 1) tmem_dealloc(tbase, 512);
}

size_t bwd_scratch_bytes(const glacore_problem *p) {
  const int64_t BT = p->B * p->T;
  return (size_t)BT * p->H * KD * sizeof(float) + (size_t)p->n_seqs * p->H * KD * sizeof(float) + 256;
}

cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO,
                const float *dht, void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws,
                cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
  BwdMaps maps;
  const int64_t BT = pr.BT;
  if (!make_map(&maps.q, pr.q, true, KD, pr.Hqk, BT, 64) ||
      !make_map(&maps.k, pr.k, true, KD, pr.Hqk, BT, 64) ||
      !make_map(&maps.v, pr.v, true, VD, pr.H, BT, 64) ||
      !make_map(&maps.dO, dO, true, VD, pr.H, BT, 64))
    return cudaErrorInvalidValue;
  BwdArgs a;
  a.docs = docs;
  a.H = pr.H;
  a.scale = pr.scale;
  a.g = pr.g;
  a.h0 = pr.h0;
  a.dht = dht;
  a.dq = (__nv_bfloat16 *)dq;
  a.dk = (__nv_bfloat16 *)dk;
  a.dv = (__nv_bfloat16 *)dv;
  a.dg = dg;
  a.dh0 = dh0;
  a.dgp = (float *)ws;
  a.bvec = (float *)(ws + (size_t)BT * pr.H * KD * sizeof(float));
  a.err = pr.err;
  dim3 grid((unsigned)docs.n, (unsigned)pr.H);
  const int smA = asm_::BYTES + 1024, smB = bsm::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(gla_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smA);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gla_bwd_rev_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smB);
  if (e != cudaSuccess) return e;
  gla_bwd_dq_kernel<<<grid, 448, smA, st>>>(maps, a);
  mark_launch("gla_bwd_dq_kernel", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gla_bwd_rev_kernel<<<grid, 448, smB, st>>>(maps, a);
  mark_launch("gla_bwd_rev_kernel", st);
  (void)p;
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace glacore
