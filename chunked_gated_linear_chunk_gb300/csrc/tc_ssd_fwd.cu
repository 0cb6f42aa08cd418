// tc_ssd_fwd.cu -- forward kernel of the SSD tcgen05 path (formulas in
// tc_ssd.cuh).
//
// One CTA per (document, head): a one-dimensional grid of units x H CTAs
// (x = rank H + head, units in launch order, longest first for packed
// batches), 512 threads, one CTA per SM.  The CTA walks its document's
// chunks in order:
//   warp 0       TMA producer (3-stage ring of q, k, v tiles)
//   warp 1       TMEM owner and MMA issuer
//   warps 2..5   mask warpgroup: the decayed, masked P as bf16 hi / lo
//                tiles
//   warps 6..9   state warpgroup: S (fp32 in registers, thread c holds
//                channel row c), bf16 copy of S for the next readout
//   warps 10..13 output warpgroup: o = scale exp(G_t) (q S)_t + (P v)_t,
//                and two chunks ahead v scaled by exp(Gam - G_s)
//   warps 14, 15 gate warps: up to two chunks ahead, the prefix sums G and
//                every decay factor of the chunk (one slot of a 3-slot
//                ring)
// TMEM (512 columns): QK[2] at 0/64, U[2] at 128/192, QS[2] at 256/320,
// PV[2] at 384/448 (M = 64 tiles: row r in lane 32 (r / 16) + r % 16).
#include "tc_ssd.cuh"

namespace glacore {
namespace ssd {

using namespace tc;

struct FwdMaps {
  CUtensorMap q, k, v;
};

struct FwdArgs {
  Units units;
  int64_t H;
  int32_t hq_div;  // heads per q / k head
  float scale;
  const float *g;   // [BT, H]
  const float *h0;  // [n_docs, H, K, V] or null
  float *ht;        // [n_docs, H, K, V] or null
  __nv_bfloat16 *o; // [BT, H, V]
  int *err;
};

namespace ffs {  // shared-memory carve-up (bytes)
constexpr int NS = 3;
constexpr uint32_t Q = 0;          // 3 x 16 KB (two 64-channel blocks of 64 tokens)
constexpr uint32_t K = 49152;      // 3 x 16 KB
constexpr uint32_t V = 98304;      // 3 x 8 KB
constexpr uint32_t VT = 122880;    // 2 x 8 KB: v (.) exp(Gam - G_s)
constexpr uint32_t P = 139264;     // 2 x 16 KB: masked P, bf16 hi (+0) and lo (+8 KB)
constexpr uint32_t S = 172032;     // 2 x 16 KB: S as bf16 (rows = channel)
constexpr uint32_t GS = 204800;    // gsl::NG gate slots
constexpr uint32_t BYTES = GS + gsl::NG * gsl::GSLOT;
}  // namespace ffs

__global__ void __launch_bounds__(512, 1) ssd_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs a) {
  using namespace ffs;
  using namespace gsl;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[NS], empty[NS], gready[NG], gfree[NG], qk_full[2], u_full[2], qs_full[2], pv_full[2],
      p_ready[2], s_ready[2], o_free[2], vt_ready[2], drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

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
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < NG; ++i) {
      mbar_init(&gready[i], 64);
      mbar_init(&gfree[i], 384);  // mask, state and output warpgroups
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&qk_full[i], 1);
      mbar_init(&u_full[i], 1);
      mbar_init(&qs_full[i], 1);
      mbar_init(&pv_full[i], 1);
      mbar_init(&p_ready[i], 128);
      mbar_init(&s_ready[i], 128);
      mbar_init(&o_free[i], 128);
      mbar_init(&vt_ready[i], 128);
    }
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
#define SSD_FAIL            \
  {                         \
    atomicExch(&abort_flag, 1); \
    break;                  \
  }
  auto tQK = [&](int b) { return tbase + 64u * b; };
  auto tU = [&](int b) { return tbase + 128u + 64u * b; };
  auto tQS = [&](int b) { return tbase + 256u + 64u * b; };
  auto tPV = [&](int b) { return tbase + 384u + 64u * b; };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      int issued = 0;
      for (int j = 0; j < nch; ++j) {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(&empty[s], ((j / NS) - 1) & 1, WAIT_CYCLES)) SSD_FAIL
        if (*abortp) break;
        const int tok = (int)chunk_tok(j);
        mbar_expect_tx(&full[s], 16384 + 16384 + 8192);
        tma_load_3d(sm + Q + s * 16384, &maps.q, 0, hq, tok, &full[s]);
        tma_load_3d(sm + Q + s * 16384 + 8192, &maps.q, 64, hq, tok, &full[s]);
        tma_load_3d(sm + K + s * 16384, &maps.k, 0, hq, tok, &full[s]);
        tma_load_3d(sm + K + s * 16384 + 8192, &maps.k, 64, hq, tok, &full[s]);
        tma_load_3d(sm + V + s * 8192, &maps.v, 0, h, tok, &full[s]);
        // the tiles of chunk j + 2 into L2: their load is issued about two
        // chunk periods from now, once a stage frees up
        if (j + 2 < nch) {
          const int tp = (int)chunk_tok(j + 2);
          tma_prefetch_3d(&maps.q, 0, hq, tp);
          tma_prefetch_3d(&maps.q, 64, hq, tp);
          tma_prefetch_3d(&maps.k, 0, hq, tp);
          tma_prefetch_3d(&maps.k, 64, hq, tp);
          tma_prefetch_3d(&maps.v, 0, h, tp);
        }
        issued = j + 1;
      }
      // every load issued has landed before the CTA leaves
      for (int j = max(0, issued - NS); j < issued; ++j)
        if (!mbar_wait(&full[j % NS], (j / NS) & 1, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // Order per chunk j: QK(j+1) as soon as its tiles land, then q_j S_{j-1},
    // then (P v)_j after the mask step, then U(j+1) = k^T vt after the gate
    // step of j+1; the next mask step finds its QK ready.
    if (lane == 0) {
      constexpr uint32_t idQK = idesc_bf16(64, 64, false, false);
      constexpr uint32_t idO = idesc_bf16(64, 64, false, true);
      constexpr uint32_t idU = idesc_bf16(128, 64, true, true);
      auto issue_qk = [&](int jj) {
        const int s = jj % NS;
        const uint32_t qa = sbase + Q + s * 16384, ka = sbase + K + s * 16384;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tQK(jj & 1), kdesc(qa, ks, 64), kdesc(ka, ks, 64), idQK, ks);
        mma_commit(&qk_full[jj & 1]);
      };
      auto issue_u = [&](int jj) {
        const uint32_t ka = sbase + K + (jj % NS) * 16384, vt = sbase + VT + (jj & 1) * 8192;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tU(jj & 1), mdesc(ka, ks, 8192), mdesc(vt, ks, 8192), idU, ks);
        mma_commit(&u_full[jj & 1]);
      };
      if (nch > 0) {
        bool ok = mbar_wait(&full[0], 0, WAIT_CYCLES);
        tc_fence_after();
        if (ok) issue_qk(0);
        ok = ok && mbar_wait(&vt_ready[0], 0, WAIT_CYCLES);
        tc_fence_after();
        if (ok) issue_u(0);
        if (!ok) atomicExch(&abort_flag, 1);
      }
      for (int j = 0; j < nch && !*abortp; ++j) {
        const int b = j & 1, s = j % NS;
        if (j + 1 < nch) {
          if (!mbar_wait(&full[(j + 1) % NS], ((j + 1) / NS) & 1, WAIT_CYCLES)) SSD_FAIL
          tc_fence_after();
          issue_qk(j + 1);
        }
        // S_{j-1} (buffer (j - 1) & 1; the entering state is in buffer 1),
        // and QS / PV buffer b read out by the output step of j - 2
        if (!mbar_wait(&s_ready[(j + 1) & 1], (j >> 1) & 1, WAIT_CYCLES)) SSD_FAIL
        if (j >= 2 && !mbar_wait(&o_free[b], ((j - 2) >> 1) & 1, WAIT_CYCLES)) SSD_FAIL
        tc_fence_after();
        {
          const uint32_t qa = sbase + Q + s * 16384, Sa = sbase + S + ((j + 1) & 1) * 16384;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) mma_bf16(tQS(b), kdesc(qa, ks, 64), mdesc(Sa, ks, 16384), idO, ks);
          mma_commit(&qs_full[b]);
        }
        if (!mbar_wait(&p_ready[b], (j >> 1) & 1, WAIT_CYCLES)) SSD_FAIL
        tc_fence_after();
        {
          const uint32_t Pa = sbase + P + b * 16384, va = sbase + V + s * 8192;
          // (P_hi + P_lo) v: the decayed P carried at about 16 bits
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tPV(b), kdesc(Pa, ks, 64), mdesc(va, ks, 8192), idO, ks);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) mma_bf16(tPV(b), kdesc(Pa + 8192, ks, 64), mdesc(va, ks, 8192), idO, 1);
          mma_commit(&pv_full[b]);
          mma_commit(&empty[s]);
        }
        if (j + 1 < nch) {
          // U's buffer (j + 1) & 1 was read by the state step of j - 1 (s_ready above); vt of j + 1 written
          if (!mbar_wait(&vt_ready[(j + 1) & 1], ((j + 1) >> 1) & 1, WAIT_CYCLES)) SSD_FAIL
          tc_fence_after();
          issue_u(j + 1);
        }
      }
      // every product issued has completed before TMEM is released
      mma_commit(&drain);
      if (!mbar_wait(&drain, 0, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else if (warp < 6) {
    // ---------------- mask warpgroup ----------------
    const int qw = warp & 3;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    for (int t = 0; t < 4; ++t) mask_tile_init(sm + P + t * 8192, qw, lane);
    bool ok = true;
    for (int j = 0; j < nch && !*abortp; ++j) {
      const int bb = j & 1, gsl = j % NG;
      // P's buffer bb was read by (P v)_{j-2}, which completed before QK(j)
      if (!mbar_wait(&qk_full[bb], (j >> 1) & 1, WAIT_CYCLES) || !mbar_wait(&gready[gsl], (j / NG) & 1, WAIT_CYCLES)) {
        ok = false;
        break;
      }
      tc_fence_after();
      decay_mask<true>(tQK(bb), lane_off, qw, lane, sm + P + bb * 16384, sm + P + bb * 16384 + 8192, slot_of(j));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&p_ready[bb]);
      mbar_arrive(&gfree[gsl]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
  } else if (warp < 10) {
    // ---------------- state warpgroup ----------------
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
    store_state_row(sm + S + 16384, c, Sr);  // the entering state, read by QS(0)
    fence_async_smem();
    mbar_arrive(&s_ready[1]);
    bool ok = true;
    for (int j = 0; j < nch && !*abortp; ++j) {
      const int bb = j & 1;
      // U(j); the gates of j; and S's buffer bb, last read by q_{j-1} S_{j-2}
      if (!mbar_wait(&u_full[bb], (j >> 1) & 1, WAIT_CYCLES) ||
          !mbar_wait(&gready[j % NG], (j / NG) & 1, WAIT_CYCLES) ||
          (j >= 1 && !mbar_wait(&qs_full[(j - 1) & 1], ((j - 1) >> 1) & 1, WAIT_CYCLES))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float eGam = lds_f1(smem_u32(slot_of(j)) + 4u * G_EGAM);
#pragma unroll
      for (int cp = 0; cp < 64; cp += 32) {
        uint32_t r[32];
        tmem_ld32(tU(bb) + lane_off + cp, r);
        tmem_ld_wait32(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) Sr[cp + i] = fmaf(eGam, Sr[cp + i], __uint_as_float(r[i]));
      }
      store_state_row(sm + S + bb * 16384, c, Sr);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&s_ready[bb]);
      mbar_arrive(&gfree[j % NG]);
    }
    if (!ok) atomicExch(&abort_flag, 1);
    if (a.ht && un.piece == un.npieces - 1 && !*abortp) {
      float *dst = a.ht + ((d * H + h) * KD + c) * VD;
#pragma unroll
      for (int i = 0; i < 64; i += 4) *reinterpret_cast<float4 *>(dst + i) = make_float4(Sr[i], Sr[i + 1], Sr[i + 2], Sr[i + 3]);
    }
  } else if (warp < 14) {
    // ---------------- output warpgroup ----------------
    const int qw = warp & 3, rl = lane & 15, row = qw * 16 + rl;
    const bool second = lane >= 16;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    // o = scale exp(G_t) (q S)_t + (P v)_t.  Lanes 0..15 hold rows
    // 16 qw .. 16 qw + 15 of the M = 64 tiles; lanes 16..31 take columns
    // 32..63 of the same rows (shuffled over), lanes 0..15 columns 0..31.
    auto output = [&](int jj) -> bool {
      const int bb = jj & 1;
      if (!mbar_wait(&qs_full[bb], (jj >> 1) & 1, WAIT_CYCLES) || !mbar_wait(&pv_full[bb], (jj >> 1) & 1, WAIT_CYCLES) ||
          !mbar_wait(&gready[jj % NG], (jj / NG) & 1, WAIT_CYCLES))
        return false;
      tc_fence_after();
      const float eg = lds_f1(smem_u32(slot_of(jj)) + 4u * (G_EG + row));
      const int L = chunk_len(jj);
      __nv_bfloat16 *orow = a.o + ((chunk_tok(jj) + row) * H + h) * VD;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint32_t xa[16], xb[16], pa[16], pb[16];
        tmem_ld16(tQS(bb) + lane_off + 16 * k, xa);
        tmem_ld16(tQS(bb) + lane_off + 32 + 16 * k, xb);
        tmem_ld16(tPV(bb) + lane_off + 16 * k, pa);
        tmem_ld16(tPV(bb) + lane_off + 32 + 16 * k, pb);
        tmem_ld_wait(xa);
        tmem_tie(xb);
        tmem_tie(pa);
        tmem_tie(pb);
        float y[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t xs = __shfl_sync(0xffffffffu, xb[i], rl), ps = __shfl_sync(0xffffffffu, pb[i], rl);
          const float x = __uint_as_float(second ? xs : xa[i]), pv = __uint_as_float(second ? ps : pa[i]);
          y[i] = fmaf(eg, x, pv);
        }
        if (row < L) {
          __nv_bfloat16 *dst = orow + (second ? 32 : 0) + 16 * k;
          st_global_v4(dst, pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                       pack_bf16(y[6], y[7]));
          st_global_v4(dst + 8, pack_bf16(y[8], y[9]), pack_bf16(y[10], y[11]), pack_bf16(y[12], y[13]),
                       pack_bf16(y[14], y[15]));
        }
      }
      tc_fence_before();
      mbar_arrive(&o_free[bb]);
      return true;
    };
    // vt = v (.) exp(Gam - G_s) of chunk jj: thread row t, 32 of its 64 columns
    auto make_vt = [&](int jj) -> bool {
      const int bb = jj & 1, s = jj % NS;
      // the gate step of jj, v of jj, and vt's buffer (read by U(jj - 2))
      if (!mbar_wait(&gready[jj % NG], (jj / NG) & 1, WAIT_CYCLES) || !mbar_wait(&full[s], (jj / NS) & 1, WAIT_CYCLES) ||
          (jj >= 2 && !mbar_wait(&u_full[bb], ((jj - 2) >> 1) & 1, WAIT_CYCLES)))
        return false;
      const int tid = (int)threadIdx.x - 320, t = tid >> 1, cb = (tid & 1) * 32;
      const float egr = lds_f1(smem_u32(slot_of(jj)) + 4u * (G_EGR + t));
      const uint32_t src = smem_u32(sm + V + s * 8192), dst = smem_u32(sm + VT + bb * 8192);
#pragma unroll
      for (int c = cb; c < cb + 32; c += 8) {
        const uint32_t off = sw128_off(t, c, 64);
        const uint4 x = lds_u4(src + off);
        st_shared_v4(dst + off, scale_bf16x2(x.x, egr), scale_bf16x2(x.y, egr), scale_bf16x2(x.z, egr),
                     scale_bf16x2(x.w, egr));
      }
      fence_async_smem();
      mbar_arrive(&vt_ready[bb]);
      return true;
    };
    bool ok = true;
    for (int jj = 0; ok && jj < 2 && jj < nch; ++jj) ok = make_vt(jj);
    for (int j = 0; ok && j < nch && !*abortp; ++j) {
      ok = output(j);
      mbar_arrive(&gfree[j % NG]);
      if (ok && j + 2 < nch) ok = make_vt(j + 2);
    }
    if (!ok) atomicExch(&abort_flag, 1);
  } else {
    // ---------------- gate warps ----------------
    const int tid = (int)threadIdx.x - 448;  // 0..63: token / row of the chunk
    // thread tid owns token tid of the chunk; its gates of the next two
    // chunks are loaded ahead
    auto load_g = [&](int jj) -> float {
      if (jj >= nch || tid >= chunk_len(jj)) return 0.f;
      return ldg_early(a.g + (chunk_tok(jj) + tid) * H + h);
    };
    float gnext = load_g(0), gnext2 = load_g(1);
    // the gate slot of chunk jj
    auto prep = [&](int jj) -> bool {
      const int gsl = jj % NG, L = chunk_len(jj);
      float *gs = slot_of(jj);
      // the slot was last read by the mask, state and output steps of jj - NG
      bool good = true;
      if (jj >= NG && !mbar_wait(&gfree[gsl], ((jj / NG) - 1) & 1, WAIT_CYCLES)) good = false;
      const int t = tid;
      const float gt = gnext;
      gnext = gnext2;
      gnext2 = load_g(jj + 2);
      float egr, eg;
      gate_factors(gs, t, lane, L, a.scale, gt, 2, egr, eg);
      (void)egr;
      (void)eg;
      if (!good) return false;
      mbar_arrive(&gready[gsl]);
      return true;
    };
    // the 64 threads leave the loop together (gate_factors holds named
    // barriers): a failed wait only stops the loop at the next chunk
    bool ok = true;
    for (int j = 0; j < nch; ++j) {
      if (named_bar_any(2, 64, !ok || *abortp)) break;
      ok = prep(j) && ok;
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
// host side
// =========================================================================

bool supported(const glacore_problem *p) {
  return p->dtype == GLACORE_BF16 && p->K == KD && p->V == VD && p->H % p->Hqk == 0 &&
         (p->q_stride % 8) == 0 && (p->k_stride % 8) == 0 && (p->v_stride % 8) == 0 &&
         (p->chunk_size == 0 || p->chunk_size == 64) && p->B * p->T < ((int64_t)1 << 31) &&
         p->n_seqs * p->H < ((int64_t)1 << 31);
}

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t workspace_bytes(const glacore_problem *p, bool backward) {
  if (backward) return bwd_workspace_bytes(p);
  size_t off = 0;
  if (p->segment_ids) off = al256(off + (size_t)p->n_seqs * sizeof(int32_t));  // launch order
  return off;
}

static Units doc_units(const Docs &docs, char *ws) {
  Units us;
  memset(&us, 0, sizeof(us));
  us.docs = docs;
  us.order = docs.start ? (const int32_t *)ws : nullptr;
  return us;
}

cudaError_t fwd(const Prob &pr, const Docs &docs, const glacore_problem *p, void *o, float *ht, char *ws,
                cudaStream_t st) {
  if (docs.n == 0) return cudaSuccess;
  if (const cudaError_t be = bind_context()) return be;
  FwdMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (!make_map(&maps.q, pr.q, true, KD, pr.Hqk, pr.BT, 64, pr.qs) ||
      !make_map(&maps.k, pr.k, true, KD, pr.Hqk, pr.BT, 64, pr.ks) ||
      !make_map(&maps.v, pr.v, true, VD, pr.H, pr.BT, 64, pr.vs))
    return cudaErrorInvalidValue;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.units = doc_units(docs, ws);
  a.H = pr.H;
  a.hq_div = (int32_t)(pr.H / pr.Hqk);
  a.scale = pr.scale;
  a.g = pr.g;
  a.h0 = pr.h0;
  a.ht = ht;
  a.o = (__nv_bfloat16 *)o;
  a.err = pr.err;
  cudaError_t e;
  if (a.units.order && (e = launch_order_units(a.units, docs.n, (int32_t *)ws, st)) != cudaSuccess) return e;
  const int smem = ffs::BYTES + 1024;
  if ((e = cudaFuncSetAttribute(ssd_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  ssd_fwd_kernel<<<(unsigned)(docs.n * pr.H), 512, smem, st>>>(maps, a);
  mark_launch("ssd_fwd_kernel", st);
  return cudaGetLastError();
}

}  // namespace ssd
}  // namespace glacore
