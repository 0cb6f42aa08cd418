// tc_gla_fwd.cuh -- the forward kernel body of the tcgen05 path for GLA with bf16 inputs,
// K = V = 128, chunk C = 64.
//
// Chunk formulas (FLAT blog, trainstation-project.github.io/blog/flat:
// "Linear Attention / Forward Recurrence" for the chunkwise form, "Gated
// Linear Attention" for the decay ratios as exponentiated chunk-local
// prefix sums of the log gate, "Backward Recurrence" / "Backward Kernels"
// for the reverse chunk walk and the gate gradient as a suffix sum):
//
//   G   = inclusive prefix sum of g over the chunk (per key channel, fp32)
//   qt  = scale q exp(G)      kt = k exp(-G)       Gam = G at the chunk end
//   P   = (qt kt^T) masked to s <= t
//   O   = qt S + P V          S <- diag(exp(Gam)) (S + kt^T V)
//
// The masked P enters P V as two bf16 tiles, hi = bf16(P) and
// lo = bf16(P - hi), so that its own rounding does not add to the error of
// o (which is rounded to bf16 once more when it is stored).
//
// The fp32 state S never leaves the SM between chunks (FLAT's "keep the
// state on-chip"; FLA instead writes every chunk state to HBM).  All
// matrix products run on tcgen05 (bf16 operands from shared memory,
// fp32 accumulators in TMEM); q/k/v/g tiles arrive by TMA.
//
// Thread roles in every kernel: warp 0 issues TMA loads (one lane), warp 1
// owns TMEM and issues tcgen05.mma (one lane), warps 2..5 are the compute
// warpgroup.  Compute thread i of the warpgroup owns key channel (or value
// column) c = 32 * (warp % 4) + lane, which is also the TMEM lane it may
// read: M = 128 accumulators are laid out one row per lane, so products
// whose rows are channels (state update, transposed gradients) land in the
// thread that owns that channel.  M = 64 accumulators (the C x C matrices,
// the output tile) put row r in lane 32 * (r / 16) + r % 16.
#pragma once

#include "tc_common.cuh"

namespace glacore {
namespace tc {

// =========================================================================
// Forward: a one-dimensional grid of 2 x units x H CTAs (a unit is a
// document or a piece of one; x = 2 (rank H + head) + value half, units in
// launch order), 448 threads, clusters of two CTAs along x.  One CTA owns
// one unit, one head and 64 value columns and walks the unit's chunks in
// order; the two CTAs of a cluster (the value halves) split the gate / q / k
// prep by key channel and exchange the prepared tiles through distributed
// shared memory.  SSD runs the same kernel with one gate per head, q / k
// shared by a group of heads and V = 64 read as 128 columns (FwdArgs:
// gate_head, hq_div, vd).
//   warp 0      TMA producer (ring of q, k, v tiles; no L2 prefetches: issued
//               from this thread they delayed the tile loads behind them)
//   warp 1      TMEM owner and MMA issuer
//   warps 2..9  prep: gates loaded ahead of their chunk, prefix/suffix products,
//               scaled q / k in place
//   warps 10..13 epilogue: causal mask of P, state update S (fp32, in
//               registers, thread c holds row c), output stores
// TMEM (512 columns): P[2] at 0/64, U[2] at 128/192, O[2] at 256/320.
// =========================================================================
struct FwdMaps {
  CUtensorMap q, k, v, g;
};
struct FwdArgs {
  Units units;
  int64_t H;
  int32_t hq_div;     // heads per q / k head (q, k are [BT, H / hq_div, K]); 0 or 1: one each
  int32_t gate_head;  // 1: g is [BT, H], one log-decay per head for all key channels
  int32_t vd;         // value columns of v and o (64 or 128); the kernels compute 128,
                      // reading v's missing columns as zeros (TMA fill)
  float scale;
  const float *g;
  const float *h0;    // [n_docs,H,K,V] state entering the document, or null
  float *ht;          // [n_docs,H,K,V] final state (written by the last piece)
  float *lbuf;        // [units,H,K,V] piece end state from zero (written by the piece pass)
  float *dbuf;        // [units,H,K] exp(sum of g over the piece) (written by the piece pass)
  int32_t all_units;  // piece pass: every unit contributes (state entries), not only pieces that hand on
  __nv_bfloat16 *o;   // [BT, H, vd]
  int *err;
};

namespace fsm {  // shared-memory carve-up of the forward kernel (bytes)
constexpr int NS = 4;             // q/k/v pipeline stages
constexpr uint32_t Q = 0;         // 4 x 16 KB: q, then qt in place
constexpr uint32_t K = 65536;     // 4 x 16 KB: k, then kt in place
constexpr uint32_t V = 131072;    // 4 x 8 KB (64 value columns)
// masked P as bf16 hi (+0) and lo (+8 KB) tiles (K-major A).  One buffer:
// the mask step of chunk j writes it only after P(j) has landed, whose
// commit follows the P V products of chunk j - 1 that read it.
constexpr uint32_t P = 163840;
constexpr uint32_t S = 180224;    // 2 x 16 KB: S (bf16, rows = key channel)
constexpr uint32_t GAM = 212992;  // 8 x 128 fp32: exp(chunk gate total), ring over chunks
constexpr int NGAM = 8;
constexpr uint32_t XCH = 217088;  // 8 KB: token-group gate products (two buffers per prep group)
constexpr uint32_t BYTES = 225280;
}  // namespace fsm

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Prep of one chunk by the prep threads of one CTA of a pair.  The two CTAs
// (value halves) of a (unit, head) share the q / k tiles: CTA `rank`
// prepares key channels 64 rank .. 64 rank + 63 (one 64-column block of
// each tile) in place; the block is then copied to the peer.
// Thread (token group pw, lane) owns channels c0, c0+1 (c0 = 64 rank +
// 2 lane) and tokens t0 = TPT pw .. t0 + TPT - 1; x holds their gates.
// exp(G_t) comes by prefix products and exp(Gam - G_t) by suffix products,
// one exponential per element; the token groups exchange their products
// through xch.
// accum (the piece passes of piece_state_kernel): the k-slot tile is scaled for a
// product accumulated over the whole piece instead of a per-chunk state
// step: with dec = (dec0, dec1) the decay of the channels over the chunks
// already visited, it becomes k exp(Gam - G) dec (forward pass, chunks
// visited last to first: the decay from each token to the piece end), or,
// when rev, holds q and becomes scale q exp(G) dec (reverse pass, chunks
// first to last: the decay from the piece start to each token).  Returns
// exp(Gam) of the two channels.
// Packed fp32 pairs (the thread's two channels): one mul.rn.f32x2 per pair,
// rounded exactly as two scalar multiplies.
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n mul.rn.f32x2 z, x, y;\n"
      " mov.b64 {%0, %1}, z;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
// TPT tokens per thread: the 64 tokens of the chunk are 64 / TPT token
// groups (tg), whose threads (bar_threads of them) meet at named barrier
// bar_id to exchange their products through xch ([64 / TPT][128] floats).
template <int TPT = 8>
__device__ __forceinline__ float2 prep_chunk_pair(uint32_t q, uint32_t k, float2 (&x)[TPT], float *gam, float *xch,
                                                int pw, int lane, int rank, int L, float scale, bool with_q,
                                                bool rev, bool accum = false,
                                                float2 dec = make_float2(1.f, 1.f), int bar_id = 1,
                                                int bar_threads = 256) {
  constexpr int NG = 64 / TPT;
  const int c0 = 64 * rank + 2 * lane;
  const int t0 = TPT * pw;
  const float2 one = make_float2(1.f, 1.f);
  float2 p = one;
#pragma unroll
  for (int i = 0; i < TPT; ++i) {
    x[i] = (t0 + i < L) ? make_float2(__expf(x[i].x), __expf(x[i].y)) : one;
    p = mul2(p, x[i]);
  }
  *reinterpret_cast<float2 *>(xch + pw * 128 + c0) = p;
  named_bar(bar_id, bar_threads);
  float2 pre = one, suf = one;
#pragma unroll
  for (int u = 0; u < NG; ++u) {
    const float2 e = *reinterpret_cast<const float2 *>(xch + u * 128 + c0);
    if (u < pw)
      pre = mul2(pre, e);
    else if (u > pw)
      suf = mul2(suf, e);
  }
  const float2 T = mul2(mul2(pre, p), suf);  // exp(Gam)
  // byte offsets of rows t0 .. t0+7 of the column pair (c0, c0+1) in a tile
  uint32_t off[TPT];
  {
    const uint32_t b = (uint32_t)(c0 >> 6) * 8192u + (uint32_t)t0 * 128u + (uint32_t)(c0 & 7) * 2u;
    const uint32_t cch = (uint32_t)(c0 & 63) >> 3;
#pragma unroll
    for (int i = 0; i < TPT; ++i) off[i] = b + ((cch ^ (uint32_t)(i & 7)) << 4) + (uint32_t)i * 128u;
  }
  const float2 sc2 = make_float2(scale, scale);
  uint32_t v[TPT];
  if (with_q) {
    float2 a = mul2(sc2, pre);
#pragma unroll
    for (int i = 0; i < TPT; ++i) v[i] = lds_u32(q + off[i]);
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      a = mul2(a, x[i]);
      const float2 r = mul2(bf2_to_f2(v[i]), a);
      v[i] = (t0 + i < L) ? pack_bf16(r.x, r.y) : 0u;
    }
#pragma unroll
    for (int i = 0; i < TPT; ++i) sts_u32(q + off[i], v[i]);
  }
  const float2 rT = accum ? dec : make_float2(__frcp_rn(T.x), __frcp_rn(T.y));
  if (!rev) {
    float2 a = mul2(suf, rT);
#pragma unroll
    for (int i = 0; i < TPT; ++i) v[i] = lds_u32(k + off[i]);
#pragma unroll
    for (int i = TPT - 1; i >= 0; --i) {
      const float2 r = mul2(bf2_to_f2(v[i]), a);
      v[i] = (t0 + i < L) ? pack_bf16(r.x, r.y) : 0u;
      a = mul2(a, x[i]);
    }
#pragma unroll
    for (int i = 0; i < TPT; ++i) sts_u32(k + off[i], v[i]);
  } else {
    float2 a = mul2(mul2(sc2, pre), rT);
#pragma unroll
    for (int i = 0; i < TPT; ++i) v[i] = lds_u32(k + off[i]);
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      a = mul2(a, x[i]);
      const float2 r = mul2(bf2_to_f2(v[i]), a);
      v[i] = (t0 + i < L) ? pack_bf16(r.x, r.y) : 0u;
    }
#pragma unroll
    for (int i = 0; i < TPT; ++i) sts_u32(k + off[i], v[i]);
  }
  if (pw == 0 && !accum) {
    gam[c0] = T.x;
    gam[c0 + 1] = T.y;
  }
  return T;
}

__device__ __forceinline__ void store_state_bf16(uint8_t *St, int c, const float (&S)[64]) {
#pragma unroll
  for (int n = 0; n < 64; n += 8)
    st_shared_v4(smem_u32(St + sw128_off(c, n, 128)), pack_bf16(S[n], S[n + 1]),
                 pack_bf16(S[n + 2], S[n + 3]), pack_bf16(S[n + 4], S[n + 5]),
                 pack_bf16(S[n + 6], S[n + 7]));
}

// HG: one gate per head (g is [BT, H]); the per-channel instance has none of
// its branches.
template <bool HG>
__device__ __forceinline__ void gla_fwd_body(const FwdMaps &maps, const FwdArgs &a, unsigned bx) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[fsm::NS], empty[fsm::NS], prep_done[fsm::NS], p_full[2], u_full[2],
      o_full[2], p_ready[2], s_ready[2], gam_ready[fsm::NGAM];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag, range_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the two value halves of a (unit, head) are a cluster of two CTAs that
  // share the q / k prep (rank = value half)
  // bx = 2 (r H + h) + vb: launch rank r (units in launch order), head h
  const int vb = bx & 1, h = (int)((int64_t)(bx >> 1) % a.H);
  const int hq = a.hq_div > 1 ? h / a.hq_div : h;  // head of q and k
  const uint32_t peer = (uint32_t)(vb ^ 1);
  const int64_t u = a.units.at((int64_t)(bx >> 1) / a.H);
  const Unit un = a.units.get(u);
  const int64_t d = un.doc;
  const int64_t s0 = un.start, s1 = un.end;
  const bool last_piece = un.piece == un.npieces - 1;
  const int nch = (int)((s1 - s0 + C - 1) / C);
  auto chunk_tok = [&](int j) -> int64_t { return s0 + (int64_t)j * C; };

  if (warp == 1) {
    tmem_alloc(&tmem_base, 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    range_flag = 0;
    for (int i = 0; i < fsm::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2);        // the MMA commits of both CTAs (multicast)
      mbar_init(&prep_done[i], 129);  // the 128 prep threads of the chunk's group + the peer's
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&u_full[i], 1);
      mbar_init(&o_full[i], 1);
      mbar_init(&p_ready[i], 128);
      mbar_init(&s_ready[i], 128);
    }
    for (int i = 0; i < fsm::NGAM; ++i) mbar_init(&gam_ready[i], 129);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
#define FAIL_AND_BREAK        \
  {                           \
    atomicExch(&abort_flag, 1); \
    break;                    \
  }

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&maps.q);
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      if (!HG) tma_prefetch_desc(&maps.g);
      for (int j = 0; j < nch; ++j) {
        const int s = j % fsm::NS;
        if (j >= fsm::NS && !mbar_wait(&empty[s], ((j / fsm::NS) - 1) & 1, WAIT_CYCLES))
          FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)chunk_tok(j);
        // this CTA's half of the q / k channels (the peer writes the other
        // half of the prepared tiles) and its value half of v
        mbar_expect_tx(&full[s], 3 * 8192);
        uint8_t *q = sm + fsm::Q + s * 16384, *k = sm + fsm::K + s * 16384;
        tma_load_3d(q + vb * 8192, &maps.q, 64 * vb, hq, tok, &full[s]);
        tma_load_3d(k + vb * 8192, &maps.k, 64 * vb, hq, tok, &full[s]);
        tma_load_3d(sm + fsm::V + s * 8192, &maps.v, vb * 64, h, tok, &full[s]);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idP = idesc_bf16(64, 64, false, false);
      constexpr uint32_t idO = idesc_bf16(64, 64, false, true);
      constexpr uint32_t idU = idesc_bf16(128, 64, true, true);
      uint32_t ph_prep = 0, ph_pr = 0, ph_sr = 0;  // one parity bit per buffer
      // Issue order: while chunk j's causal mask is being applied, the
      // products of chunk j + 1 that need no state (P, and U once the
      // state step of j - 1 has read U's tile) and q_j S_{j-1} are already
      // running, so that after the mask step only the two P V products stand
      // between it and the output tile, and the next mask step finds its P.
      // (The epilogue writes the masked P of chunk j + 1 into the one P tile
      // only after it has stored output j, so P V of chunk j has read it.)
      auto issue_p = [&](int jj) -> bool {  // P of chunk jj, once it is prepared
        const int sj = jj % fsm::NS;
        if (!mbar_wait_cluster(&prep_done[sj], (ph_prep >> sj) & 1, WAIT_CYCLES)) return false;
        ph_prep ^= 1u << sj;
        tc_fence_after();
        const uint32_t qa = sbase + fsm::Q + sj * 16384, ka = sbase + fsm::K + sj * 16384;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tbase + 64 * (jj & 1), kdesc(qa, ks, 64), kdesc(ka, ks, 64), idP, ks);
        mma_commit(&p_full[jj & 1]);
        return true;
      };
      auto issue_u = [&](int jj) {  // U = kt^T v of chunk jj
        const int sj = jj % fsm::NS;
        const uint32_t ka = sbase + fsm::K + sj * 16384, va = sbase + fsm::V + sj * 8192;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tbase + 128 + 64 * (jj & 1), mdesc(ka, ks, 8192), mdesc(va, ks, 8192), idU, ks);
        mma_commit(&u_full[jj & 1]);
      };
      if (nch > 0) {
        if (issue_p(0))
          issue_u(0);
        else
          atomicExch(&abort_flag, 1);
      }
      for (int j = 0; j < nch && !*abortp; ++j) {
        const int b = j & 1, st = j % fsm::NS;
        const uint32_t qa = sbase + fsm::Q + st * 16384, va = sbase + fsm::V + st * 8192;
        const uint32_t Pa = sbase + fsm::P, Sa = sbase + fsm::S + (b ^ 1) * 16384;
        const uint32_t tO = tbase + 256 + 64 * b;
        const bool next = j + 1 < nch;
        if (next && !issue_p(j + 1)) FAIL_AND_BREAK
        // S_{j-1} in shared memory; U's tile (j + 1) & 1 read by its state step
        if (!mbar_wait(&s_ready[b ^ 1], (ph_sr >> (b ^ 1)) & 1, WAIT_CYCLES)) FAIL_AND_BREAK
        ph_sr ^= 1u << (b ^ 1);
        tc_fence_after();
        if (next) issue_u(j + 1);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) mma_bf16(tO, kdesc(qa, ks, 64), mdesc(Sa, ks, 16384), idO, ks);
        if (!mbar_wait(&p_ready[b], (ph_pr >> b) & 1, WAIT_CYCLES)) FAIL_AND_BREAK
        ph_pr ^= 1u << b;
        tc_fence_after();
        // P V as (P_hi + P_lo) V: the masked P carried at about 16 bits
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tO, kdesc(Pa, ks, 64), mdesc(va, ks, 8192), idO, 1);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) mma_bf16(tO, kdesc(Pa + 8192, ks, 64), mdesc(va, ks, 8192), idO, 1);
        mma_commit(&o_full[b]);
        mma_commit_multicast(&empty[st], 3);
      }
      // every commit that targets this CTA's stage barriers has landed
      // before the CTAs leave (the peer's arrive on our barriers and ours on
      // its): wait for the last phase of each stage
      for (int j = max(0, nch - fsm::NS); j < nch && !*abortp; ++j)
        if (!mbar_wait(&empty[j % fsm::NS], (j / fsm::NS) & 1, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else if (warp < 10) {
    // ---------------- prep warps (8) ----------------
    // Two groups of four warps take alternate chunks (group g: chunks j with
    // j % 2 == g), so that two chunks' prep chains are in flight at once.
    // Thread: this CTA's key channels c0, c0 + 1, tokens 16 tg .. 16 tg + 15.
    const int pw = warp - 2, grp = pw >> 2, tg = pw & 3;
    const int c0 = 64 * vb + 2 * lane, t0 = 16 * tg;
    const uint32_t rem = mapa_shared(sbase, peer);  // the peer's tiles
    // gates of the group's next chunk are loaded while this one is prepared
    float2 xn[16];
    auto load_x = [&](int jj, float2 (&x)[16]) {
      const int64_t tk = chunk_tok(jj);
      const int LL = (int)min((int64_t)C, s1 - tk);
      if constexpr (HG) {  // one gate per head: the same for both channels
        const float *gp = a.g + (tk + t0) * a.H + h;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float gv = (t0 + i < LL) ? ldg_early(gp + (int64_t)i * a.H) : 0.f;
          x[i] = make_float2(gv, gv);
        }
      } else {
        const float *gp = a.g + ((tk + t0) * a.H + h) * KD + c0;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          x[i] = (t0 + i < LL) ? ldg_early2(gp + (int64_t)i * a.H * KD) : make_float2(0.f, 0.f);
      }
    };
    if (grp < nch) load_x(grp, xn);
    for (int j = grp; j < nch; j += 2) {
      const int s = j % fsm::NS;
      const int64_t tok0 = chunk_tok(j);
      const int L = (int)min((int64_t)C, s1 - tok0);
      float2 x[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = xn[i];
      if (j + 2 < nch) load_x(j + 2, xn);
      if (!mbar_wait(&full[s], (j / fsm::NS) & 1, WAIT_CYCLES)) FAIL_AND_BREAK
      // this CTA's 64-column block of q, k and its gate totals (byte offsets)
      const uint32_t qo = fsm::Q + s * 16384 + vb * 8192, ko = fsm::K + s * 16384 + vb * 8192,
                     go = fsm::GAM + (j % fsm::NGAM) * 512 + vb * 256;
      const float2 gam = prep_chunk_pair<16>(
          sbase + fsm::Q + s * 16384, sbase + fsm::K + s * 16384, x,
          reinterpret_cast<float *>(sm + fsm::GAM + (j % fsm::NGAM) * 512),
          reinterpret_cast<float *>(sm + fsm::XCH) + (2 * grp + ((j >> 1) & 1)) * 512, tg, lane, vb, L, a.scale,
          true, false, false, make_float2(1.f, 1.f), 1 + grp, 128);
      // decay outside the range of the chunk-local factorisation (NaN too)
      if (tg == 0 && !(fminf(gam.x, gam.y) >= kMinChunkDecay)) range_flag = 1;
      fence_async_smem();
      // copy the prepared blocks into the peer's tiles (bulk copies that
      // complete on the peer's barriers; one arrive there stands for the
      // 128 threads of the group here)
      named_bar(1 + grp, 128);
      if (tg == 0 && lane == 0) {
        const uint32_t pbar = mapa_shared(smem_u32(&prep_done[s]), peer);
        const uint32_t gbar = mapa_shared(smem_u32(&gam_ready[j % fsm::NGAM]), peer);
        mbar_arrive_expect_tx_cluster(pbar, 16384u);
        bulk_copy_to_cluster(rem + qo, sbase + qo, 8192, pbar);
        bulk_copy_to_cluster(rem + ko, sbase + ko, 8192, pbar);
        mbar_arrive_expect_tx_cluster(gbar, 256u);
        bulk_copy_to_cluster(rem + go, sbase + go, 256, gbar);
      }
      mbar_arrive(&prep_done[s]);
      mbar_arrive(&gam_ready[j % fsm::NGAM]);
    }
  } else {
    // ---------------- epilogue warpgroup ----------------
    const int qw = warp & 3;
    const int c = qw * 32 + lane;       // key channel = TMEM lane of M = 128 tiles
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    const int prow = qw * 16 + lane;    // row of M = 64 tiles (lanes < 16)
    const int64_t H = a.H;
    const int v0 = vb * 64;
    float S[64];
    {
      // state entering the unit: h0 folded over the document's earlier pieces
      const float *h0row = a.h0 ? a.h0 + ((d * H + h) * KD + c) * VD : nullptr;
      piece_state_in<64>(S, h0row, a.lbuf, a.dbuf, u - un.piece, un.piece, H, h, c, v0);
    }
    for (int t = 0; t < 2; ++t) mask_tile_init(sm + fsm::P + t * 8192, qw, lane);
    store_state_bf16(sm + fsm::S + 16384, c, S);
    fence_async_smem();
    mbar_arrive(&s_ready[1]);
    uint32_t ph_p = 0, ph_u = 0, ph_o = 0;
    for (int j = 0; j < nch; ++j) {
      const int b = j & 1;
      const int64_t tok0 = chunk_tok(j);
      const int L = (int)min((int64_t)C, s1 - tok0);
      const uint32_t tP = tbase + 64 * b, tU = tbase + 128 + 64 * b, tO = tbase + 256 + 64 * b;
      // S2: P -> causal mask -> bf16 hi / lo A operands of the intra-chunk product
      if (!mbar_wait(&p_full[b], (ph_p >> b) & 1, WAIT_CYCLES)) {
        FAIL_AND_BREAK
      }
      ph_p ^= 1u << b;
      tc_fence_after();
      mask_tile_to_smem_hilo(tP, lane_off, qw, lane, sm + fsm::P, sm + fsm::P + 8192);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&p_ready[b]);
      // S3a: state update S <- exp(Gam) (S + kt^T V), bf16 copy for the next readout
      if (!mbar_wait(&u_full[b], (ph_u >> b) & 1, WAIT_CYCLES) ||
          !mbar_wait_cluster(&gam_ready[j % fsm::NGAM], (j / fsm::NGAM) & 1, WAIT_CYCLES)) {
        FAIL_AND_BREAK
      }
      ph_u ^= 1u << b;
      tc_fence_after();
      const float eG = reinterpret_cast<const float *>(sm + fsm::GAM)[(j % fsm::NGAM) * 128 + c];
#pragma unroll
      for (int cp = 0; cp < 4; cp += 2) {
        uint32_t r[16], r2[16];
        tmem_ld16(tU + lane_off + cp * 16, r);
        tmem_ld16(tU + lane_off + cp * 16 + 16, r2);
        tmem_ld_wait(r);
        tmem_tie(r2);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          S[cp * 16 + i] = eG * (S[cp * 16 + i] + __uint_as_float(r[i]));
          S[cp * 16 + 16 + i] = eG * (S[cp * 16 + 16 + i] + __uint_as_float(r2[i]));
        }
      }
      store_state_bf16(sm + fsm::S + b * 16384, c, S);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&s_ready[b]);
      // S3b: output tile O = qt S_prev + P V
      if (!mbar_wait(&o_full[b], (ph_o >> b) & 1, WAIT_CYCLES)) {
        FAIL_AND_BREAK
      }
      ph_o ^= 1u << b;
      tc_fence_after();
#pragma unroll
      for (int cp = 0; cp < 4; cp += 2) {
        uint32_t r[2][16];
        tmem_ld16(tO + lane_off + cp * 16, r[0]);
        tmem_ld16(tO + lane_off + cp * 16 + 16, r[1]);
        tmem_ld_wait(r[0]);
        tmem_tie(r[1]);
        // o has 128 columns, or in the per-head-gate instance a.vd (64 or
        // 128): a value half at or past them stores nothing
        const int Lo = (!HG || (int)(blockIdx.x & 1) * 64 < a.vd) ? L : 0;
        if (lane < 16 && prow < Lo) {
#pragma unroll
          for (int hc = 0; hc < 2; ++hc) {
            __nv_bfloat16 *dst = a.o + ((tok0 + prow) * H + h) * (HG ? (int64_t)a.vd : (int64_t)VD) + v0 + (cp + hc) * 16;
            const uint32_t *x = r[hc];
            st_global_v4(dst, pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                         pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                         pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                         pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
            st_global_v4(dst + 8, pack_bf16(__uint_as_float(x[8]), __uint_as_float(x[9])),
                         pack_bf16(__uint_as_float(x[10]), __uint_as_float(x[11])),
                         pack_bf16(__uint_as_float(x[12]), __uint_as_float(x[13])),
                         pack_bf16(__uint_as_float(x[14]), __uint_as_float(x[15])));
          }
        }
      }
      tc_fence_before();
    }
    float *dst = a.ht && last_piece ? a.ht + ((d * H + h) * KD + c) * VD + v0 : nullptr;
    if (dst && !*abortp) {
#pragma unroll
      for (int n = 0; n < 64; n += 4)
        *reinterpret_cast<float4 *>(dst + n) = make_float4(S[n], S[n + 1], S[n + 2], S[n + 3]);
    }
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync();  // no remote access to this CTA's shared memory after this point
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (range_flag && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_RANGE);
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace tc
}  // namespace glacore
