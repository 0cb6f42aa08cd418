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
// as M = 128 tcgen05 accumulators, so the thread that reads row c of TMEM
// owns channel c for the suffix sums.  Thread roles: warp 0 TMA, warp 1
// MMA + TMEM owner, warps 2..9 per-channel warps (thread = one key channel
// x 32 tokens; gate work, exp(+-G) staged in their own TMEM lanes, and in
// pass B the dk / dv / dg epilogue), warps 10..13 masks and the state; in
// pass A warps 14..17 run the dq epilogue (thread = one key channel, all 64
// tokens).  SSD runs the same kernels with one
// gate per head, q / k shared by a group of heads and V = 64 read as 128
// columns (BwdArgs: gate_head, hq_div, vd).
#include <string.h>

#include "tc_gla_fwd.cuh"

namespace glacore {
namespace tc {

struct BwdMaps {
  CUtensorMap q, k, v, dO, dq, g, dk, dv, qt, kt;
};
struct BwdArgs {
  Units units;
  int64_t H;
  int32_t hq_div;     // heads per q / k head (q, k are [BT, H / hq_div, K]); 0 or 1: one each
  int32_t gate_head;  // 1: g is [BT, H], one log-decay per head for all key channels
  int32_t vd;         // value columns of v, do and dv (64 or 128); the kernels compute
                      // 128, reading the missing columns as zeros
  float scale;
  const float *g;
  const float *h0;     // [n_docs,H,K,V] or null
  const float *dht;    // [n_docs,H,K,V] or null
  __nv_bfloat16 *dq, *dk, *dv;
  float *dg, *dh0;
  float *dgp;    // scratch [chunk slots, H, C/4, K, 4] fp32: within-chunk suffix sums of q (.) dq
  float *bvec;   // scratch [units, H, K] fp32
  const float *lf, *df;  // forward piece hand-off: [units,H,K,V] end states from zero, [units,H,K] decays
  const float *lr, *dr;  // reverse piece hand-off: [units,H,K,V] state gradients at the piece
                         // starts from zero at their ends, [units,H,K] decays
  float *ckpt;   // [slots, H, V/4, K, 4] fp32 state every CKPT_CHUNKS chunks (pass A -> pass B)
  __nv_bfloat16 *qt, *kt;  // scratch [BT, H, K]: gated q and k (pass A -> pass B)
  uint16_t *eng;  // scratch [chunk slots, H, C/4, K, 4] bf16: exp(-G) (pass A -> pass B)
  float *egam;    // scratch [chunk slots, H, K] fp32: each chunk's exp(-Gam) exactly, for the
                  // state-gradient recurrence (pass A -> pass B)
  int *err;
};

// Global chunk index of local chunk 0 of a unit (document chunk base plus
// the piece's offset inside its document).
__device__ __forceinline__ int64_t unit_chunk0(const Units &us, const Unit &un) {
  int64_t ds, de;
  us.docs.range(un.doc, ds, de);
  return us.docs.chunk_base(un.doc) + (un.start - ds) / C;
}
// Checkpoint slot of the boundary after global chunk gc, or -1.  Slots are
// floor(gc / CKPT_CHUNKS): boundaries of one document are CKPT_CHUNKS chunks
// apart and documents are disjoint chunk ranges, so slots never collide.
__device__ __forceinline__ int64_t ckpt_slot(int64_t gc0, int64_t doc_c0, int j, int nch) {
  if (j >= nch - 1) return -1;  // the unit's end uses the piece / document boundary term
  const int64_t jd = gc0 - doc_c0 + j;  // chunk index inside the document
  if ((jd + 1) % CKPT_CHUNKS) return -1;
  return (gc0 + j) / CKPT_CHUNKS;
}

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
    cg.x[i] = t < L ? ldg_early(g + ((tok0 + t) * H + h) * KD + c) : 0.f;
  }
}
__device__ __forceinline__ void load_gates_to(float (&x)[32], const float *g, int64_t tok0, int64_t H,
                                              int h, int c, int th, int L) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int t = 32 * th + i;
    x[i] = t < L ? ldg_early(g + ((tok0 + t) * H + h) * KD + c) : 0.f;
  }
}
// Tokens 32 th + I0 .. 32 th + I0 + N - 1 of load_gates_to: the loads of one
// chunk are issued in parts so that fewer misses are in flight at once.
template <int I0, int N>
__device__ __forceinline__ void load_gates_part(float (&x)[32], const float *g, int64_t tok0, int64_t H,
                                                int h, int c, int th, int L) {
#pragma unroll
  for (int i = I0; i < I0 + N; ++i) {
    const int t = 32 * th + i;
    x[i] = t < L ? ldg_early(g + ((tok0 + t) * H + h) * KD + c) : 0.f;
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
constexpr uint32_t Q = 0;          // 2 x 16 KB raw q, then dq in place (store source)
constexpr uint32_t K = 32768;      // 2 x 16 KB k, then kt in place
constexpr uint32_t V = 65536;      // 2 x 16 KB
constexpr uint32_t DO = 98304;     // 2 x 16 KB
constexpr uint32_t DP = 131072;    // 8 KB masked dP (bf16 [t][s])
constexpr uint32_t GT = 139264;    // 2 x 32 KB gate tiles g [t][c] (fp32, TMA box 32 x 64)
constexpr uint32_t QT = 204800;    // 16 KB qt = scale q exp(G) (bf16, store source for pass B)
constexpr uint32_t XCH = 221184;   // 2 x 2 x 128 fp32 gate products
constexpr uint32_t BYTES = 223232;
}  // namespace asm_

// Thread roles: warp 0 lane 0 TMA loads of k, v, do; lane 1 TMA loads of
// raw q; lane 2 TMA stores of dq and qt; lane 3 TMA loads of the gate tile
// (per-channel gates; a per-head gate is staged by 64 of the per-channel
// threads instead); lane 4 TMA stores of kt.  Pass B takes the gated
// operands qt, kt from here instead of gating q and k again.  Warp 1
// MMA + TMEM.  Warps 2..9 per-channel warps (key channel c = lane of the
// warp's TMEM quarter, token half th): gate work and kt of each chunk.
// Warps 10..13 mask dP and scale the state.  Warps 14..17 the dq / q (.) dq
// epilogue (key channel c, all tokens of the chunk), written to shared
// memory for the TMA stores, so that it overlaps the next chunk's gate work.
// HG: one gate per head (g is [BT, H]); the per-channel instance has none of
// its branches.
template <bool HG>
__global__ void __launch_bounds__(576, 1)
    gla_bwd_dq_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[asm_::NS], empty[asm_::NS], qfull[asm_::NS], qempty[asm_::NS],
      prep_done[asm_::NS], dp_full, dp_ready, dq_full[2], dq_free[2], u_full, s_ready, eg_ready[2],
      eg_free[2], out_ready, stg_free, g_full[2], g_free[2], kt_read[asm_::NS];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, range_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // blockIdx.x = r H + h: launch rank r (units in launch order), head h
  const int h = (int)((int64_t)blockIdx.x % a.H);
  const int64_t u = a.units.at((int64_t)blockIdx.x / a.H);
  const int64_t H = a.H;
  const Unit un = a.units.get(u);
  const int64_t d = un.doc;
  const int64_t s0 = un.start, s1 = un.end;
  const int nch = (int)((s1 - s0 + C - 1) / C);
  const int hq = a.hq_div > 1 ? h / a.hq_div : h;  // head of q and k

  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    range_flag = 0;
    for (int i = 0; i < asm_::NS; ++i) {
      mbar_init(&full[i], 1);    // k, v, do (released by the MMA commit)
      mbar_init(&empty[i], 1);
      mbar_init(&qfull[i], 1);   // raw q, then dq (released by the store thread)
      mbar_init(&qempty[i], 1);
      mbar_init(&prep_done[i], 256);
      mbar_init(&kt_read[i], 1);  // kt of the stage copied out (lane 4)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&dq_full[i], 1);
      mbar_init(&dq_free[i], 128);   // epilogue warps
      mbar_init(&eg_ready[i], 256);
      mbar_init(&eg_free[i], 256);   // state and epilogue warps
    }
    mbar_init(&dp_full, 1);
    mbar_init(&dp_ready, 128);
    mbar_init(&u_full, 1);
    mbar_init(&s_ready, 128);
    mbar_init(&out_ready, 128);
    mbar_init(&stg_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&g_full[i], 1);
      mbar_init(&g_free[i], 256);
    }
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
  // TMEM columns: dP, S_prev (bf16 A operand), dq^T[2], S, exp(G)[2]
  const uint32_t tDP = tbase, tSb = tbase + 64, tDQ = tbase + 128, tS = tbase + 256, tEG = tbase + 384;

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      tma_prefetch_desc(&maps.dO);
      if (!HG) tma_prefetch_desc(&maps.g);
      for (int j = 0; j < nch; ++j) {
        const int st = j % asm_::NS;
        if (j >= asm_::NS && (!mbar_wait(&empty[st], ((j / asm_::NS) - 1) & 1, WAIT_CYCLES) ||
                              !mbar_wait(&kt_read[st], ((j / asm_::NS) - 1) & 1, WAIT_CYCLES)))
          BW_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)(s0 + (int64_t)j * C);
        mbar_expect_tx(&full[st], 3 * 16384);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(sm + asm_::K + st * 16384 + x * 8192, &maps.k, 64 * x, hq, tok, &full[st]);
          tma_load_3d(sm + asm_::V + st * 16384 + x * 8192, &maps.v, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + asm_::DO + st * 16384 + x * 8192, &maps.dO, 64 * x, h, tok, &full[st]);
        }
      }
    } else if (lane == 1) {
      tma_prefetch_desc(&maps.q);
      for (int j = 0; j < nch; ++j) {
        const int st = j % asm_::NS;
        if (j >= asm_::NS && !mbar_wait(&qempty[st], ((j / asm_::NS) - 1) & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)(s0 + (int64_t)j * C);
        mbar_expect_tx(&qfull[st], 16384);
        for (int x = 0; x < 2; ++x)
          tma_load_3d(sm + asm_::Q + st * 16384 + x * 8192, &maps.q, 64 * x, hq, tok, &qfull[st]);
      }
    } else if (lane == 2) {
      // stores of full chunks (a ragged chunk is stored by its epilogue threads)
      tma_prefetch_desc(&maps.dq);
      tma_prefetch_desc(&maps.qt);
      for (int j = 0; j < nch; ++j) {
        const int st = j % asm_::NS;
        const int64_t tok0 = s0 + (int64_t)j * C;
        if (!mbar_wait(&out_ready, j & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        if (s1 - tok0 >= C) {
          for (int x = 0; x < 2; ++x) {
            tma_store_3d(&maps.dq, sm + asm_::Q + st * 16384 + x * 8192, 64 * x, h, (int)tok0);
            tma_store_3d(&maps.qt, sm + asm_::QT + x * 8192, 64 * x, h, (int)tok0);
          }
          bulk_commit();
          bulk_wait_read_all();
        }
        mbar_arrive(&qempty[st]);
        mbar_arrive(&stg_free);
      }
      bulk_wait_all();
    } else if (lane == 3 && !HG) {
      // gate tile of each chunk (two buffers: chunk j's tile is loaded once
      // the prep has read chunk j-2's)
      for (int j = 0; j < nch; ++j) {
        const int gb = j & 1;
        if (j >= 2 && !mbar_wait(&g_free[gb], ((j >> 1) - 1) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)(s0 + (int64_t)j * C);
        mbar_expect_tx(&g_full[gb], 32768);
        for (int x = 0; x < 4; ++x)
          tma_load_3d(sm + asm_::GT + gb * 32768 + x * 8192, &maps.g, 32 * x, h, tok, &g_full[gb]);
      }
    } else if (lane == 4) {
      // kt of each full chunk to the workspace once the prep has written it
      // (a ragged chunk is stored by the prep threads); the stage is
      // refilled only after this copy has read it
      tma_prefetch_desc(&maps.kt);
      uint32_t ph = 0;
      for (int j = 0; j < nch; ++j) {
        const int st = j % asm_::NS;
        const int64_t tok0 = s0 + (int64_t)j * C;
        if (!mbar_wait(&prep_done[st], (ph >> st) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph ^= 1u << st;
        if (s1 - tok0 >= C) {
          for (int x = 0; x < 2; ++x)
            tma_store_3d(&maps.kt, sm + asm_::K + st * 16384 + x * 8192, 64 * x, h, (int)tok0);
          bulk_commit();
          bulk_wait_read_all();
        }
        mbar_arrive(&kt_read[st]);
      }
      bulk_wait_all();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idDP = idesc_bf16(64, 64, false, false);
      constexpr uint32_t idU = idesc_bf16(128, 128, true, true);
      constexpr uint32_t idQ1 = idesc_bf16(128, 64, false, false);
      constexpr uint32_t idQ2 = idesc_bf16(128, 64, true, false);
      const uint32_t dpa = sbase + asm_::DP;
      uint32_t ph_prep = 0, ph_dqf = 0;
      for (int j = 0; j < nch; ++j) {
        const int st = j % asm_::NS, b = j & 1;
        const uint32_t ka = sbase + asm_::K + st * 16384, va = sbase + asm_::V + st * 16384;
        const uint32_t doa = sbase + asm_::DO + st * 16384;
        if (!mbar_wait(&prep_done[st], (ph_prep >> st) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph_prep ^= 1u << st;
        tc_fence_after();
        // dP = dO V^T  (the mask of chunk j-1 has read tDP: dq^T(j-1) waited for it)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tDP, kdesc(doa, ks, 64), kdesc(va, ks, 64), idDP, ks);
        mma_commit(&dp_full);
        // S (TMEM, = S_prev) += kt^T V
        if (!mbar_wait(&s_ready, j & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tS, mdesc(ka, ks, 8192), mdesc(va, ks, 8192), idU, 1);
        mma_commit(&u_full);
        // dq^T = S_prev dO^T + kt^T dP^T  (dq^T buffer b free once chunk j-2 is read)
        if (!mbar_wait(&dp_ready, j & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        if (j >= 2) {
          if (!mbar_wait(&dq_free[b], (ph_dqf >> b) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
          ph_dqf ^= 1u << b;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16_ta(tDQ + 64 * b, tSb + 8 * ks, kdesc(doa, ks, 64), idQ1, ks);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tDQ + 64 * b, mdesc(ka, ks, 8192), kdesc(dpa, ks, 64), idQ2, 1);
        mma_commit(&dq_full[b]);
        mma_commit(&empty[st]);
      }
    }
  } else if (warp < 10) {
    // ---------- per-channel warps: key channel c, tokens 32 th .. +31 ----------
    const int qw = warp & 3, th = (warp - 2) >> 2;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    const int64_t gc0 = unit_chunk0(a.units, un);
    uint32_t ph_full = 0, ph_free = 0;
    const ColF32 gcol(sbase + asm_::GT, 32 * th, c);  // buffer 0; buffer 1 is 32 KB on
    // one gate per head: thread (th = 0, c < 64) fetches token c's gate two
    // chunks ahead and stages it in the gate buffer of its chunk before the
    // exchange barrier of the chunk before (gate of token t at byte 4 t)
    const bool stager = HG && th == 0 && c < C;
    auto gate_of = [&](int jj) -> float {
      const int64_t t0 = s0 + (int64_t)jj * C;
      return (jj < nch && t0 + c < s1) ? ldg_early(a.g + (t0 + c) * H + h) : 0.f;
    };
    float gnext = 0.f;
    if (stager) {
      reinterpret_cast<float *>(sm + asm_::GT)[c] = gate_of(0);
      gnext = gate_of(1);
    }
    if (HG) named_bar(1, 256);
    // gate work and kt of chunk j
    for (int j = 0; j < nch; ++j) {
      {
        const int st = j % asm_::NS, b = j & 1;
        const int64_t tok0 = s0 + (int64_t)j * C;
        const int L = (int)min((int64_t)C, s1 - tok0);
        ChanGate cg;
        if constexpr (HG) {
          // the gates of chunk j (the same for every channel), staged two chunks
          // ago; the next chunk's go to the other buffer before this chunk's
          // exchange barrier, and the one after next is fetched
          const uint32_t gs = sbase + asm_::GT + b * 32768 + 128 * th;
#pragma unroll
          for (int i = 0; i < 32; ++i) cg.x[i] = lds_f32(gs + 4 * i);
          if (stager) {
            reinterpret_cast<float *>(sm + asm_::GT + (b ^ 1) * 32768)[c] = gnext;
            gnext = gate_of(j + 2);
          }
        } else {
          if (!mbar_wait(&g_full[b], (j >> 1) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
#pragma unroll
          for (int i = 0; i < 32; ++i) cg.x[i] = 32 * th + i < L ? lds_f32(gcol.at(i) + b * 32768) : 0.f;
          mbar_arrive(&g_free[b]);
        }
        if (!mbar_wait(&full[st], (ph_full >> st) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        ph_full ^= 1u << st;
        exchange_gates(cg, reinterpret_cast<float *>(sm + asm_::XCH) + b * 256, c, th, L);
        // decay outside the range of the chunk-local factorisation (NaN too)
        if (th == 0 && !(cg.total >= kMinChunkDecay)) range_flag = 1;
        // exp(G_t) -> TMEM (dq scaling; column 63 = exp(Gam) for the state step)
        if (j >= 2) {
          if (!mbar_wait(&eg_free[b], (ph_free >> b) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
          ph_free ^= 1u << b;
        }
        tc_fence_after();
        {
          float pre = cg.before;
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              pre *= cg.x[16 * hb + i];
              r[i] = __float_as_uint(pre);
            }
            tmem_st16(tEG + 64 * b + lane_off + 32 * th + 16 * hb, r);
          }
        }
        // kt = k exp(-Gam) exp(Gam - G) in place
        {
          const ColBf16 kc(sbase + asm_::K + st * 16384, 32 * th, c);
          float sc = cg.after * __frcp_rn(cg.total);
#pragma unroll
          for (int hb = 1; hb >= 0; --hb) {
            uint16_t kb[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) kb[i] = lds_u16(kc.at(16 * hb + i));
            float en[16];  // exp(-G_t)
#pragma unroll
            for (int i = 15; i >= 0; --i) {
              const int t = 32 * th + 16 * hb + i;
              en[i] = sc;
              kb[i] = f32_to_bf16_bits(t < L ? bf16_bits_to_f32(kb[i]) * sc : 0.f);
              sc *= cg.x[16 * hb + i];
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) sts_u16(kc.at(16 * hb + i), kb[i]);
            {
              // exp(-G) for pass B in bf16 (it scales dk, which is rounded
              // to bf16 in turn), chunk-slot layout as the partials: four
              // tokens of one channel per 8 bytes; the chunk's exp(-Gam)
              // (token 63) also in fp32, for the state-gradient recurrence
              uint2 *dst = reinterpret_cast<uint2 *>(a.eng) + ((gc0 + j) * H + h) * (int64_t)(KD * C / 4) + c;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[(8 * th + 4 * hb + q) * KD] =
                    make_uint2(pack_bf16(en[4 * q], en[4 * q + 1]), pack_bf16(en[4 * q + 2], en[4 * q + 3]));
              if (th == 1 && hb == 1) a.egam[((gc0 + j) * H + h) * KD + c] = en[15];
            }
            if (L < C) {  // ragged chunk: kt rows < L straight to the workspace
              const int tb = 32 * th + 16 * hb;
              float kv[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) kv[i] = bf16_bits_to_f32(kb[i]);
              transpose_4x4_blocks(kv, lane);
              store_block_bf16(a.kt + ((tok0 + tb) * H + h) * KD + 32 * qw, H * KD, kv, lane, tb, L);
            }
          }
        }
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&prep_done[st]);
        mbar_arrive(&eg_ready[b]);
      }
    }
  } else if (warp < 14) {
    // ---------------- state warpgroup: thread = key channel c ----------------
    const int qw = warp & 3;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    mask_tile_init(sm + asm_::DP, qw, lane);
    // S (TMEM) = state entering the unit (h0 folded over the document's
    // earlier pieces), bf16 copy (TMEM A operand) for chunk 0's readout
    {
      const float *h0row = a.h0 ? a.h0 + ((d * H + h) * KD + c) * VD : nullptr;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float sv[32];
        piece_state_in<32>(sv, h0row, a.lf, a.df, u - un.piece, un.piece, H, h, c, 32 * cb);
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(sv[i]);
        tmem_st32(tS + lane_off + 32 * cb, r);
        uint32_t pk[16];
#pragma unroll
        for (int n = 0; n < 16; ++n) pk[n] = pack_bf16(sv[2 * n], sv[2 * n + 1]);
        tmem_st16(tSb + lane_off + 16 * cb, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s_ready);
    }
    uint32_t ph_egr = 0, ph_dqf = 0;
    const int64_t gc0 = unit_chunk0(a.units, un), doc_c0 = a.units.docs.chunk_base(un.doc);
    for (int j = 0; j < nch; ++j) {
      const int b = j & 1;
      // (1) masked dP -> bf16 operand (dq^T of chunk j-1, its last reader, is
      //     complete: dp_full(j) is committed after it)
      if (!mbar_wait(&dp_full, j & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      tc_fence_after();
      mask_tile_to_smem(tDP, lane_off, qw, lane, sm + asm_::DP);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&dp_ready);
      // (2) S <- exp(Gam) (S_prev + kt^T V) in TMEM; its bf16 copy replaces
      //     S_prev's once dq^T of chunk j has read that
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
        tc_fence_before();
        mbar_arrive(&eg_free[b]);
        bool waited = false;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          tmem_ld32(tS + lane_off + 32 * cb, r);
          tmem_ld_wait32(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(eGam * __uint_as_float(r[i]));
          tmem_st32(tS + lane_off + 32 * cb, r);
          if (!waited) {
            if (!mbar_wait(&dq_full[b], (ph_dqf >> b) & 1, WAIT_CYCLES)) {
              atomicExch(&abort_flag, 1);
              break;
            }
            ph_dqf ^= 1u << b;
            waited = true;
          }
          uint32_t pk[16];
#pragma unroll
          for (int n = 0; n < 16; ++n) pk[n] = pack_bf16(__uint_as_float(r[2 * n]), __uint_as_float(r[2 * n + 1]));
          tmem_st16(tSb + lane_off + 16 * cb, pk);
        }
        if (*abortp) break;
        tmem_st_wait();
        const int64_t slot = ckpt_slot(gc0, doc_c0, j, nch);
        if (slot >= 0) {
          // exact boundary state for pass B's gate-gradient carry, as
          // [value quad][channel] x 4 columns: each warp store covers 512
          // contiguous bytes
          float *dst = a.ckpt + (slot * H + h) * (int64_t)(KD * VD) + 4 * c;
#pragma unroll 1
          for (int cb = 0; cb < 8; ++cb) {
            uint32_t r[16];
            tmem_ld16(tS + lane_off + 16 * cb, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int e = 0; e < 16; e += 4)
              *reinterpret_cast<float4 *>(dst + (4 * cb + e / 4) * (4 * KD)) =
                  make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]), __uint_as_float(r[e + 2]),
                              __uint_as_float(r[e + 3]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s_ready);
    }
    // final-state term of the gate gradient: bvec = (S_end (.) dH_end) 1_V
    // (dH_end: dht folded over the document's later pieces)
    if (!*abortp && a.bvec) {
      float acc = 0.f;
      const float *dhtrow = a.dht ? a.dht + ((d * H + h) * KD + c) * VD : nullptr;
      if (dhtrow || un.piece + 1 < un.npieces) {
#pragma unroll 1
        for (int cb = 0; cb < 8; ++cb) {
          float dh[16];
          piece_grad_out<16>(dh, dhtrow, a.lr, a.dr, u - un.piece, un.piece, un.npieces, H, h, c, 16 * cb);
          uint32_t r[16];
          tmem_ld16(tS + lane_off + 16 * cb, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int i = 0; i < 16; ++i) acc += __uint_as_float(r[i]) * dh[i];
        }
      }
      a.bvec[(u * H + h) * KD + c] = acc;
    }
  } else {
    // ---------- epilogue warpgroup: key channel c, all tokens of the chunk ----------
    //   dq_t = scale exp(G_t) acc_t,  dgp_t = sum_{r >= t in chunk} q_r dq_r
    // Full chunks go to shared memory (dq over the raw q it was computed
    // from) for the TMA stores; a ragged last chunk is stored directly.
    const int qw = warp & 3;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    const int64_t gc0 = unit_chunk0(a.units, un);
    uint32_t ph_dqf = 0, ph_egr = 0;
    for (int jj = 0; jj < nch; ++jj) {
      const int bb = jj & 1, stt = jj % asm_::NS;
      const int64_t tok0 = s0 + (int64_t)jj * C;
      const int L = (int)min((int64_t)C, s1 - tok0);
      if (!mbar_wait(&dq_full[bb], (ph_dqf >> bb) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      ph_dqf ^= 1u << bb;
      if (!mbar_wait(&eg_ready[bb], (ph_egr >> bb) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      ph_egr ^= 1u << bb;
      if (!mbar_wait(&qfull[stt], (jj / asm_::NS) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      // the qt staging buffer is free once the previous chunk's stores have read it
      if (jj >= 1 && !mbar_wait(&stg_free, (jj - 1) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      tc_fence_after();
      const ColBf16 qc(sbase + asm_::Q + stt * 16384, 0, c);
      const ColBf16 qtc(sbase + asm_::QT, 0, c);
      // partials in the chunk-slot layout of the scratch: four tokens of one
      // channel per 16 bytes, [token quad][channel], so each warp store
      // covers 512 contiguous bytes (read back the same way by pass B)
      float4 *dst = reinterpret_cast<float4 *>(a.dgp) + ((gc0 + jj) * H + h) * (int64_t)(KD * C / 4) + c;
      float suf = 0.f;
#pragma unroll 1
      for (int blk = 3; blk >= 0; --blk) {
        const int tb = 16 * blk;  // first token of the block
        uint32_t acc[16], eg[16];
        tmem_ld16(tDQ + 64 * bb + lane_off + tb, acc);
        tmem_ld16(tEG + 64 * bb + lane_off + tb, eg);
        uint16_t qb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) qb[i] = lds_u16(qc.a[i & 7] + (uint32_t)(tb + i) * 128u);
        tmem_ld_wait(acc);
        tmem_ld_wait(eg);
        float dqv[16], qtv[16], sv[16];
#pragma unroll
        for (int i = 15; i >= 0; --i) {
          const float sg = a.scale * __uint_as_float(eg[i]);
          const float qf = bf16_bits_to_f32(qb[i]);
          dqv[i] = sg * __uint_as_float(acc[i]);
          qtv[i] = sg * qf;  // qt = scale q exp(G), the gated q of pass B
          if (tb + i < L) suf += qf * dqv[i];
          sv[i] = suf;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[(4 * blk + q) * KD] = make_float4(sv[4 * q], sv[4 * q + 1], sv[4 * q + 2], sv[4 * q + 3]);
        if (L == C) {
#pragma unroll
          for (int i = 0; i < 16; ++i) sts_u16(qc.a[i & 7] + (uint32_t)(tb + i) * 128u, f32_to_bf16_bits(dqv[i]));
#pragma unroll
          for (int i = 0; i < 16; ++i) sts_u16(qtc.a[i & 7] + (uint32_t)(tb + i) * 128u, f32_to_bf16_bits(qtv[i]));
        } else {
          transpose_4x4_blocks(dqv, lane);
          store_block_bf16(a.dq + ((tok0 + tb) * H + h) * KD + 32 * qw, H * KD, dqv, lane, tb, L);
          transpose_4x4_blocks(qtv, lane);
          store_block_bf16(a.qt + ((tok0 + tb) * H + h) * KD + 32 * qw, H * KD, qtv, lane, tb, L);
        }
      }
      tc_fence_before();
      mbar_arrive(&dq_free[bb]);
      mbar_arrive(&eg_free[bb]);
      fence_async_smem();
      mbar_arrive(&out_ready);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (range_flag && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_RANGE);
  if (warp == 1) tmem_dealloc(tbase, 512);
}

// ===========================================================================
// pass B
// ===========================================================================
namespace bsm {  // shared-memory carve-up (bytes)
constexpr int NS = 2;               // stages of the qt / do ring
constexpr int NK = 3;               // stages of the kt / v ring (held until dk / dv are stored)
// qt and do share a 32 KB stage, kt and v another: [qt; do] and [kt; v] are
// the 128-row operands of the stacked P / dP product.  Within a stage the
// 64-column blocks go qt (kt) block 0, do (v) block 0, qt (kt) block 1, do (v)
// block 1, 8 KB each, so either tile alone has its blocks 16 KB apart.
constexpr uint32_t QD = 0;         // 2 x 32 KB qt (gated by pass A) and do
constexpr uint32_t KV = 65536;     // 3 x 32 KB kt (gated by pass A) and v, then dk and dv (store sources)
constexpr uint32_t P = 163840;     // 8 KB masked P  (bf16 [t][s])
constexpr uint32_t DP = 172032;    // 8 KB masked dP (bf16 [t][s])
constexpr uint32_t DH = 180224;    // 32 KB dHh (bf16 [c][v])
constexpr uint32_t XK = 215040;    // 2 x 2 x 128 fp32: token-half totals of k (.) dk
constexpr uint32_t BND = 217088;   // 2 x 128 fp32: exact gate-gradient carry at checkpoints
constexpr uint32_t BYTES = 218112;
}  // namespace bsm

// Thread roles: warp 0 lane 0 TMA loads of qt, do; lane 1 TMA loads of kt,
// v; lane 2 TMA stores of dk, dv.  Warp 1 MMA + TMEM.  Warps 2..9
// per-channel warps (key channel / value column c, token half th): exp(-G)
// of chunk i (written by pass A) into TMEM, then the dk / dg / dv epilogue
// of chunk i-1, dk and dv written over kt and v for the TMA stores.  Warps
// 10..13 scale the state gradient and mask P and dP.
__device__ __forceinline__ void gla_bwd_rev_body(const BwdMaps &maps, const BwdArgs &a, unsigned bx) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[bsm::NS], empty[bsm::NS], kfull[bsm::NK], kempty[bsm::NK],
      prep_done[bsm::NS], out_ready[bsm::NK], pdp_full, pdp_ready, dh_ready, dh_full, kv_full, kv_free,
      bnd_ready[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // bx = r H + h: launch rank r (units in launch order), head h
  const int h = (int)((int64_t)bx % a.H);
  const int64_t u = a.units.at((int64_t)bx / a.H);
  const int64_t H = a.H;
  const Unit un = a.units.get(u);
  const int64_t d = un.doc;
  const int64_t s0 = un.start, s1 = un.end;
  const int nch = (int)((s1 - s0 + C - 1) / C);

  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < bsm::NS; ++i) {
      mbar_init(&full[i], 1);    // q, do: released by the MMA commit
      mbar_init(&empty[i], 1);
      mbar_init(&prep_done[i], 256);
    }
    for (int i = 0; i < bsm::NK; ++i) {
      mbar_init(&kfull[i], 1);   // kt, v (then dk, dv): released by the store thread
      mbar_init(&kempty[i], 1);
      mbar_init(&out_ready[i], 256);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bnd_ready[i], 128);
    }
    mbar_init(&pdp_full, 1);
    mbar_init(&pdp_ready, 128);
    mbar_init(&dh_ready, 128);
    mbar_init(&dh_full, 1);
    mbar_init(&kv_full, 1);
    mbar_init(&kv_free, 256);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
  // tPP: the stacked product, P in lanes 0..63 of its first 64 columns,
  // dP in lanes 64..127 of the next 64
  const uint32_t tDH = tbase, tPP = tbase + 128, tDK = tbase + 256,
                 tDV = tbase + 320, tEG = tbase + 384;
  const int64_t gc0 = unit_chunk0(a.units, un), doc_c0 = a.units.docs.chunk_base(un.doc);

  // chunks are visited in reverse: iteration i handles chunk j = nch - 1 - i
  if (warp == 0) {
    if (lane == 0) {
      // ring of q, do: released by the MMA commit
      tma_prefetch_desc(&maps.qt);
      tma_prefetch_desc(&maps.dO);
      tma_prefetch_desc(&maps.g);
      for (int i = 0; i < nch; ++i) {
        const int j = nch - 1 - i, st = i % bsm::NS;
        if (i >= bsm::NS && !mbar_wait(&empty[st], ((i / bsm::NS) - 1) & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)(s0 + (int64_t)j * C);
        mbar_expect_tx(&full[st], 2 * 16384);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(sm + bsm::QD + st * 32768 + x * 16384, &maps.qt, 64 * x, h, tok, &full[st]);
          tma_load_3d(sm + bsm::QD + st * 32768 + x * 16384 + 8192, &maps.dO, 64 * x, h, tok, &full[st]);
        }
      }
    } else if (lane == 1) {
      // ring of k and v: released once dk and dv (written over them) are stored
      tma_prefetch_desc(&maps.kt);
      tma_prefetch_desc(&maps.v);
      for (int i = 0; i < nch; ++i) {
        const int j = nch - 1 - i, st = i % bsm::NK;
        if (i >= bsm::NK && !mbar_wait(&kempty[st], ((i / bsm::NK) - 1) & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)(s0 + (int64_t)j * C);
        mbar_expect_tx(&kfull[st], 2 * 16384);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(sm + bsm::KV + st * 32768 + x * 16384, &maps.kt, 64 * x, h, tok, &kfull[st]);
          tma_load_3d(sm + bsm::KV + st * 32768 + x * 16384 + 8192, &maps.v, 64 * x, h, tok, &kfull[st]);
        }
      }
    } else if (lane == 2) {
      // dk / dv of full chunks out (a ragged chunk is stored by its epilogue
      // threads); the kt / v stage is refilled once they have been read
      tma_prefetch_desc(&maps.dk);
      tma_prefetch_desc(&maps.dv);
      for (int i = 0; i < nch; ++i) {
        const int j = nch - 1 - i, st = i % bsm::NK;
        const int64_t tok0 = s0 + (int64_t)j * C;
        if (!mbar_wait(&out_ready[st], (i / bsm::NK) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        if (s1 - tok0 >= C) {
          for (int x = 0; x < 2; ++x) {
            tma_store_3d(&maps.dk, sm + bsm::KV + st * 32768 + x * 16384, 64 * x, h, (int)tok0);
            if (64 * x < a.vd)  // dv has vd columns
              tma_store_3d(&maps.dv, sm + bsm::KV + st * 32768 + x * 16384 + 8192, 64 * x, h, (int)tok0);
          }
          bulk_commit();
          bulk_wait_read_all();
        }
        mbar_arrive(&kempty[st]);
      }
      bulk_wait_all();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idPP = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idMM = idesc_bf16(128, 64, true, true);   // MN-major A and B
      constexpr uint32_t idKK = idesc_bf16(128, 64, false, false); // K-major A and B
      constexpr uint32_t idMK = idesc_bf16(128, 64, true, false);  // MN-major A, K-major B
      constexpr uint32_t idH = idesc_bf16(128, 128, true, true);
      uint32_t ph_prep = 0;
      const uint32_t pa = sbase + bsm::P, dpa = sbase + bsm::DP, dha = sbase + bsm::DH;
      for (int i = 0; i < nch; ++i) {
        const int st = i % bsm::NS, sk = i % bsm::NK;
        const uint32_t qa = sbase + bsm::QD + st * 32768, kta = sbase + bsm::KV + sk * 32768;
        const uint32_t va = kta + 8192, doa = qa + 8192;
        if (!mbar_wait(&prep_done[st], (ph_prep >> st) & 1, WAIT_CYCLES) ||
            !mbar_wait(&full[st], (i / bsm::NS) & 1, WAIT_CYCLES) ||
            !mbar_wait(&kfull[sk], (i / bsm::NK) & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        ph_prep ^= 1u << st;
        tc_fence_after();
        // [P, .; ., dP] = [qt; dO] [kt; v]^T  (one M = 128, N = 128 product)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tPP, kdesc(qa, ks, 128), kdesc(kta, ks, 128), idPP, ks);
        mma_commit(&pdp_full);
        // dH (TMEM, = dHh after the state step) += qt^T dO
        if (!mbar_wait(&dh_ready, i & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tDH, mdesc(qa, ks, 16384), mdesc(doa, ks, 16384), idH, 1);
        mma_commit(&dh_full);
        // dk/dv accumulators are free once the epilogue of chunk i-1 has read them
        if (!mbar_wait(&pdp_ready, i & 1, WAIT_CYCLES) ||
            (i >= 1 && !mbar_wait(&kv_free, (i - 1) & 1, WAIT_CYCLES)))
          BW_FAIL_AND_BREAK
        tc_fence_after();
        // dk^T = qt^T dP + dHh V^T
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tDK, mdesc(qa, ks, 16384), mdesc(dpa, ks, 8192), idMM, ks);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tDK, kdesc(dha, ks, 128), kdesc(va, ks, 128), idKK, 1);
        // dv^T = dO^T P + dHh^T kt^T
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tDV, mdesc(doa, ks, 16384), mdesc(pa, ks, 8192), idMM, ks);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tDV, mdesc(dha, ks, 16384), kdesc(kta, ks, 128), idMK, 1);
        mma_commit(&kv_full);
        mma_commit(&empty[st]);
      }
    }
  } else if (warp < 10) {
    // ------- per-channel warps: key channel / value column c, tokens 32 th .. +31 -------
    const int qw = warp & 3, th = (warp - 2) >> 2;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    float carry = a.bvec ? a.bvec[(u * H + h) * KD + c] : 0.f;
    // exp(-G) of the next chunk (in visiting order), this half's tokens, as
    // written by pass A (bf16, chunk-slot layout: [token quad][channel] x 4)
    uint2 en4[8];
    auto load_en = [&](int jj) {
      const float *ep = reinterpret_cast<const float *>(a.eng + ((gc0 + jj) * H + h) * (int64_t)(KD * C) + 4 * c);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float2 x = ldg_early2(ep + (8 * th + w) * (2 * KD));
        en4[w] = make_uint2(__float_as_uint(x.x), __float_as_uint(x.y));
      }
    };
    if (nch > 0) load_en(nch - 1);
    // iteration i: exp(-G) of chunk nch-1-i, then the epilogue of the previous one
    for (int i = 0; i <= nch; ++i) {
      if (i < nch) {
        const int j = nch - 1 - i, st = i % bsm::NS, b = i & 1;
        const int64_t tok0 = s0 + (int64_t)j * C;
        const int L = (int)min((int64_t)C, s1 - tok0);
        // the q (.) dq partials of this chunk (read by its epilogue in the
        // next iteration) into L2: 32 KB, one 128-byte line per thread
        prefetch_l2(a.dgp + ((gc0 + j) * H + h) * (int64_t)(KD * C) + (th * 128 + c) * 32);
        uint2 e4[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) e4[w] = en4[w];
        if (j >= 1) load_en(j - 1);
        // exp(-G) -> TMEM for the dk epilogue (buffer b was last read by
        // these threads' epilogue of chunk i - 2)
        tc_fence_after();
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t r[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint2 e = e4[4 * hb + q];
            r[4 * q] = e.x << 16;
            r[4 * q + 1] = e.x & 0xffff0000u;
            r[4 * q + 2] = e.y << 16;
            r[4 * q + 3] = e.y & 0xffff0000u;
          }
          tmem_st16(tEG + 64 * b + lane_off + 32 * th + 16 * hb, r);
        }
        if (L < C) {
          // ragged chunk: the tile rows t >= L hold the next document's
          // tokens; qt and kt must be zero there
          const int sk = i % bsm::NK;
          if (!mbar_wait(&full[st], (i / bsm::NS) & 1, WAIT_CYCLES) ||
              !mbar_wait(&kfull[sk], (i / bsm::NK) & 1, WAIT_CYCLES))
            BW_FAIL_AND_BREAK
          const ColBf16 qc(sbase + bsm::QD + st * 32768, 32 * th, c, 16384);
          const ColBf16 kc(sbase + bsm::KV + sk * 32768, 32 * th, c, 16384);
#pragma unroll
          for (int w = 0; w < 32; ++w)
            if (32 * th + w >= L) {
              sts_u16(qc.at(w), 0);
              sts_u16(kc.at(w), 0);
            }
        }
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(&prep_done[st]);
      }
      if (i >= 1) {
        // epilogue of chunk jj (visited at ii = i - 1), this thread's half:
        //   dk_t = exp(-G_t) acc_t (channel c),  dv_t (value column c),
        //   dg_t = dgp_t - sum_{r >= t in chunk} k_r dk_r + carry,  k dk = kt acc
        const int ii = i - 1, jj = nch - 1 - ii, bb = ii & 1, stt = ii % bsm::NK;
        const int64_t tok0 = s0 + (int64_t)jj * C;
        const int L = (int)min((int64_t)C, s1 - tok0);
        // q (.) dq partials of channel c, this half's tokens (chunk-slot
        // layout of the scratch written by pass A: [token quad][channel] x 4
        // tokens), loaded while the products complete; the chunk's total is
        // the partial at its first token
        const float *gp = a.dgp + ((gc0 + jj) * H + h) * (int64_t)(KD * C) + 4 * c;
        float4 qp4[8];
#pragma unroll
        for (int w = 0; w < 8; ++w) qp4[w] = ldg_early4(gp + (8 * th + w) * (4 * KD));
        const float qtot = ldg_early(gp);
        if (!mbar_wait(&kv_full, ii & 1, WAIT_CYCLES) ||
            !mbar_wait(&bnd_ready[bb], (ii >> 1) & 1, WAIT_CYCLES))
          BW_FAIL_AND_BREAK
        tc_fence_after();
        // the carry restarts from the exact boundary term at a checkpoint
        const float cin = ckpt_slot(gc0, doc_c0, jj, nch) >= 0
                              ? reinterpret_cast<const float *>(sm + bsm::BND)[bb * 128 + c]
                              : carry;
        const ColBf16 kc(sbase + bsm::KV + stt * 32768, 32 * th, c, 16384);
        const ColBf16 vc(sbase + bsm::KV + stt * 32768 + 8192, 32 * th, c, 16384);
        float dgv[32];
        float sk = 0.f;
#pragma unroll
        for (int blk = 1; blk >= 0; --blk) {
          const int tb = 32 * th + 16 * blk;
          uint32_t acc[16], eg[16];
          tmem_ld16(tDK + lane_off + tb, acc);
          tmem_ld16(tEG + 64 * bb + lane_off + tb, eg);
          float qp[16];
          uint16_t kb[16];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float4 q4 = qp4[4 * blk + w];
            qp[4 * w] = q4.x;
            qp[4 * w + 1] = q4.y;
            qp[4 * w + 2] = q4.z;
            qp[4 * w + 3] = q4.w;
          }
#pragma unroll
          for (int w = 0; w < 16; ++w) kb[w] = lds_u16(kc.at(16 * blk + w));
          tmem_ld_wait(acc);
          tmem_ld_wait(eg);
          float dkv[16];
#pragma unroll
          for (int w = 15; w >= 0; --w) {
            dkv[w] = __uint_as_float(eg[w]) * __uint_as_float(acc[w]);
            sk += bf16_bits_to_f32(kb[w]) * __uint_as_float(acc[w]);  // kt is 0 past L
            dgv[16 * blk + w] = qp[w] - sk + cin;
          }
          if (L == C) {
#pragma unroll
            for (int w = 0; w < 16; ++w) sts_u16(kc.at(16 * blk + w), f32_to_bf16_bits(dkv[w]));
          } else {
            transpose_4x4_blocks(dkv, lane);
            store_block_bf16(a.dk + ((tok0 + tb) * H + h) * KD + 32 * qw, H * KD, dkv, lane, tb, L);
          }
        }
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const int tb = 32 * th + 16 * blk;
          uint32_t acc[16];
          tmem_ld16(tDV + lane_off + tb, acc);
          tmem_ld_wait(acc);
          float dvv[16];
#pragma unroll
          for (int w = 0; w < 16; ++w) dvv[w] = __uint_as_float(acc[w]);
          if (L == C) {
#pragma unroll
            for (int w = 0; w < 16; ++w) sts_u16(vc.at(16 * blk + w), f32_to_bf16_bits(dvv[w]));
          } else {
            transpose_4x4_blocks(dvv, lane);
            store_block_bf16(a.dv + ((tok0 + tb) * H + h) * a.vd + 32 * qw, H * a.vd, dvv, lane, tb, L,
                             a.vd - 32 * qw);
          }
        }
        tc_fence_before();
        mbar_arrive(&kv_free);
        // token-half totals of k (.) dk: the low half's suffixes include the high half's
        float *xk = reinterpret_cast<float *>(sm + bsm::XK) + bb * 256;
        xk[th * 128 + c] = sk;
        named_bar(2, 256);
        const float other = xk[(1 - th) * 128 + c];
        const float off = th == 0 ? other : 0.f;
        {
          // channel c of token t: each warp store covers one token's 32
          // consecutive channels (128 contiguous bytes)
          float *dgc = a.dg + ((tok0 + 32 * th) * H + h) * KD + c;
#pragma unroll
          for (int w = 0; w < 32; ++w)
            if (32 * th + w < L) dgc[(int64_t)w * H * KD] = dgv[w] - off;
        }
        carry = cin + qtot - (sk + other);
        fence_async_smem();
        mbar_arrive(&out_ready[stt]);
      }
    }
  } else {
    // ------------- state-gradient warpgroup: thread = key channel c -------------
    const int qw = warp & 3;
    const int c = 32 * qw + lane;
    const uint32_t lane_off = (uint32_t)(32 * qw) << 16;
    // lane quarters 0, 1 hold rows 0..31, 32..63 of P; quarters 2, 3 those of dP
    uint8_t *const mtile = sm + (qw < 2 ? bsm::P : bsm::DP);
    const int mr0 = 32 * (qw & 1);
    const uint32_t tM = tPP + lane_off + (qw < 2 ? 0u : 64u);
    mask_rows_init(mtile, mr0, lane);
    // dH = state gradient leaving the unit: dht folded over the document's
    // later pieces
    {
      const float *dhtrow = a.dht ? a.dht + ((d * H + h) * KD + c) * VD : nullptr;
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float dh[32];
        piece_grad_out<32>(dh, dhtrow, a.lr, a.dr, u - un.piece, un.piece, un.npieces, H, h, c, 32 * cb);
        uint32_t r[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(dh[e]);
        tmem_st32(tDH + lane_off + 32 * cb, r);
      }
      tmem_st_wait();
    }
    // each chunk's exp(-Gam) as pass A wrote it (fp32), one chunk ahead
    auto load_eg = [&](int jj) -> float { return ldg_early(a.egam + ((gc0 + jj) * H + h) * KD + c); };
    float egn = nch > 0 ? load_eg(nch - 1) : 1.f;
    for (int i = 0; i < nch; ++i) {
      const int j = nch - 1 - i, b = i & 1;
      (void)b;
      const float egc = egn;
      if (j >= 1) egn = load_eg(j - 1);
      // (1) dHh = exp(Gam) dH in TMEM; its bf16 copy replaces chunk i-1's
      //     once dk/dv of chunk i-1 have read that.  This step does not need
      //     chunk i's P and dP, so it runs while their products complete.
      if (i >= 1 && !mbar_wait(&dh_full, (i - 1) & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      tc_fence_after();
      {
        const float eGam = __frcp_rn(egc);  // 1 / exp(-Gam)
        uint8_t *Dt = sm + bsm::DH;
        const int64_t slot = ckpt_slot(gc0, doc_c0, j, nch);
        // checkpoint rows of channel c ([value quad][channel] x 4 layout)
        const float *ck = slot >= 0 ? a.ckpt + (slot * H + h) * (int64_t)(KD * VD) + 4 * c : nullptr;
        if (j >= 1) {
          // the next chunk's checkpoint (64 KB) into L2, one line per thread and quarter
          const int64_t ns = ckpt_slot(gc0, doc_c0, j - 1, nch);
          if (ns >= 0) {
            const char *nb = reinterpret_cast<const char *>(a.ckpt + ns * H * (int64_t)(KD * VD) +
                                                            h * (int64_t)(KD * VD));
#pragma unroll
            for (int x = 0; x < 4; ++x) prefetch_l2(nb + (x * 128 + c) * 128);
          }
        }
        float bnd = 0.f;
        bool waited = i == 0;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t r[32];
          float4 cv[8];
          if (ck) {
#pragma unroll
            for (int e = 0; e < 8; ++e) cv[e] = ldg_early4(ck + (8 * cb + e) * (4 * KD));
          }
          tmem_ld32(tDH + lane_off + 32 * cb, r);
          tmem_ld_wait32(r);
          if (ck) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              bnd += cv[e].x * __uint_as_float(r[4 * e]) + cv[e].y * __uint_as_float(r[4 * e + 1]) +
                     cv[e].z * __uint_as_float(r[4 * e + 2]) + cv[e].w * __uint_as_float(r[4 * e + 3]);
          }
#pragma unroll
          for (int w = 0; w < 32; ++w) r[w] = __float_as_uint(eGam * __uint_as_float(r[w]));
          tmem_st32(tDH + lane_off + 32 * cb, r);
          if (!waited) {
            if (!mbar_wait(&kv_full, (i - 1) & 1, WAIT_CYCLES)) {
              atomicExch(&abort_flag, 1);
              break;
            }
            waited = true;
          }
#pragma unroll
          for (int n = 0; n < 32; n += 8)
            st_shared_v4(smem_u32(Dt + sw128_off(c, 32 * cb + n, 128)),
                         pack_bf16(__uint_as_float(r[n]), __uint_as_float(r[n + 1])),
                         pack_bf16(__uint_as_float(r[n + 2]), __uint_as_float(r[n + 3])),
                         pack_bf16(__uint_as_float(r[n + 4]), __uint_as_float(r[n + 5])),
                         pack_bf16(__uint_as_float(r[n + 6]), __uint_as_float(r[n + 7])));
        }
        if (*abortp) break;
        tmem_st_wait();
        // exact (S_end (.) dH_end) 1_V at this boundary, for the carry
        reinterpret_cast<float *>(sm + bsm::BND)[b * 128 + c] = bnd;
        mbar_arrive(&bnd_ready[b]);
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&dh_ready);
      // (2) masked P and dP -> bf16 operands (dk/dv of chunk i-1, their last
      //     readers, are complete: pdp_full(i) is committed after them)
      if (!mbar_wait(&pdp_full, i & 1, WAIT_CYCLES)) BW_FAIL_AND_BREAK
      tc_fence_after();
      mask_rows_to_smem(tM, mr0, lane, mtile);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&pdp_ready);
    }
    // the last dH update
    if (nch > 0 && !*abortp && !mbar_wait(&dh_full, (nch - 1) & 1, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    tc_fence_after();
    float *dst = nullptr;
    if (a.dh0 && un.piece == 0) {
      dst = a.dh0 + ((d * H + h) * KD + c) * VD;
    }
    if (!*abortp && dst) {
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        uint32_t r[32];
        tmem_ld32(tDH + lane_off + 32 * cb, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int w = 0; w < 32; w += 4)
          *reinterpret_cast<float4 *>(dst + 32 * cb + w) =
              make_float4(__uint_as_float(r[w]), __uint_as_float(r[w + 1]), __uint_as_float(r[w + 2]),
                          __uint_as_float(r[w + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (warp == 1) tmem_dealloc(tbase, 512);
}

__global__ void __launch_bounds__(448)
    gla_bwd_rev_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  gla_bwd_rev_body(maps, a, blockIdx.x);
}

cudaError_t bwd(const Prob &pr, const Docs &docs, const glacore_problem *p, const void *dO,
                const float *dht, void *dq, void *dk, void *dv, float *dg, float *dh0, char *ws,
                cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
  if (const cudaError_t be = bind_context()) return be;
  const TcLayout Lo = tc_layout(p, true);
  BwdMaps maps;
  memset(&maps, 0, sizeof(maps));
  const int64_t BT = pr.BT;
  float *dgp = (float *)(ws + Lo.off_dgp);
  if (!make_map(&maps.q, pr.q, true, KD, pr.Hqk, BT, 64, pr.qs) ||
      !make_map(&maps.k, pr.k, true, KD, pr.Hqk, BT, 64, pr.ks) ||
      !make_map(&maps.v, pr.v, true, pr.V, pr.H, BT, 64, pr.vs) ||
      !make_map(&maps.dO, dO, true, pr.V, pr.H, BT, 64) ||
      !make_map(&maps.dq, dq, true, KD, pr.H, BT, 64) ||
      (!pr.gate_head && !make_map(&maps.g, pr.g, false, KD, pr.H, BT, 32)) ||
      !make_map(&maps.dk, dk, true, KD, pr.H, BT, 64) ||
      !make_map(&maps.dv, dv, true, pr.V, pr.H, BT, 64) ||
      !make_map(&maps.qt, ws + Lo.off_qt, true, KD, pr.H, BT, 64) ||
      !make_map(&maps.kt, ws + Lo.off_kt, true, KD, pr.H, BT, 64))
    return cudaErrorInvalidValue;
  BwdArgs a;
  memset(&a, 0, sizeof(a));
  a.units = units_of(docs, Lo, ws);
  a.H = pr.H;
  a.hq_div = (int32_t)(pr.H / pr.Hqk);
  a.gate_head = pr.gate_head;
  a.vd = (int32_t)pr.V;
  a.scale = pr.scale;
  a.g = pr.g;
  a.h0 = pr.h0;
  a.dht = dht;
  a.dq = (__nv_bfloat16 *)dq;
  a.dk = (__nv_bfloat16 *)dk;
  a.dv = (__nv_bfloat16 *)dv;
  a.dg = dg;
  a.dh0 = dh0;
  a.dgp = dgp;
  a.bvec = (float *)(ws + Lo.off_bvec);
  a.ckpt = (float *)(ws + Lo.off_ckpt);
  a.qt = (__nv_bfloat16 *)(ws + Lo.off_qt);
  a.eng = (uint16_t *)(ws + Lo.off_eng);
  a.egam = (float *)(ws + Lo.off_egam);
  a.kt = (__nv_bfloat16 *)(ws + Lo.off_kt);
  a.err = pr.err;
  const dim3 grid((unsigned)(Lo.max_units * pr.H));
  const int smA = asm_::BYTES + 1024, smB = bsm::BYTES + 1024;
  cudaError_t e;
  auto *dq_kernel = a.gate_head ? gla_bwd_dq_kernel<true> : gla_bwd_dq_kernel<false>;
  if ((e = cudaFuncSetAttribute(dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smA)) != cudaSuccess ||
      (e = cudaFuncSetAttribute(gla_bwd_rev_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smB)) != cudaSuccess)
    return e;
  if (Lo.pieces && Lo.table &&
      (e = launch_build_units(docs, Lo.plen, (Unit *)(ws + Lo.off_units), Lo.max_units, st)) != cudaSuccess)
    return e;
  if (a.units.order &&
      (e = launch_order_units(a.units, Lo.max_units, (int32_t *)(ws + Lo.off_order), st)) != cudaSuccess)
    return e;
  if (Lo.pieces) {
    a.lf = (const float *)(ws + Lo.off_L);
    a.df = (const float *)(ws + Lo.off_D);
    a.lr = (const float *)(ws + Lo.off_Lr);
    a.dr = (const float *)(ws + Lo.off_Dr);
    // local end states of the pieces (forward) and local state gradients at
    // their starts (reverse), in one launch; the consumers fold them
    FwdMaps fm, rm;
    memset(&fm, 0, sizeof(fm));
    if (!make_map(&fm.q, pr.q, true, KD, pr.Hqk, BT, 64, pr.qs) ||
        !make_map(&fm.k, pr.k, true, KD, pr.Hqk, BT, 64, pr.ks) ||
        !make_map(&fm.v, pr.v, true, pr.V, pr.H, BT, 64, pr.vs) ||
        (!pr.gate_head && !make_map(&fm.g, pr.g, false, KD, pr.H, BT, 32)))
      return cudaErrorInvalidValue;
    rm = fm;
    rm.k = fm.q;   // the reverse pass runs q through the k slot ...
    rm.v = maps.dO;  // ... and do through the v slot
    FwdArgs fa;
    memset(&fa, 0, sizeof(fa));
    fa.units = a.units;
    fa.H = pr.H;
    fa.hq_div = a.hq_div;
    fa.gate_head = a.gate_head;
    fa.vd = a.vd;
    fa.scale = pr.scale;
    fa.g = pr.g;
    fa.err = pr.err;
    FwdArgs ra = fa;
    fa.lbuf = (float *)(ws + Lo.off_L);
    fa.dbuf = (float *)(ws + Lo.off_D);
    ra.lbuf = (float *)(ws + Lo.off_Lr);
    ra.dbuf = (float *)(ws + Lo.off_Dr);
    if ((e = launch_piece_states(fm, fa, &rm, &ra, Lo.max_units, pr.H, st)) != cudaSuccess) return e;
  }
  dq_kernel<<<grid, 576, smA, st>>>(maps, a);
  mark_launch("gla_bwd_dq_kernel", st);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gla_bwd_rev_kernel<<<grid, 448, smB, st>>>(maps, a);
  mark_launch("gla_bwd_rev_kernel", st);
  (void)p;
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace glacore
