// tc_pieces.cu -- exact sequence split for the tensor-core kernels.
//
// A document whose (document x head) count is too small to fill the GPU is
// cut into pieces of P tokens (P a multiple of the chunk length) that run in
// parallel.  The hand-off between pieces is exact (JLA product page,
// karlex.ai/jla: "our split is exact", unlike starting every piece from
// zero): the recurrence is linear in the state, so with
//   L_p = end state of piece p started from zero,  D_p = exp(sum of g over p)
// the state entering piece p is
//   S_in[0] = h0,   S_in[p] = diag(D_{p-1}) S_in[p-1] + L_{p-1},
// and in reverse time, with Lr_p the state gradient at the start of piece p
// from its own outputs started from zero at its end,
//   dH_end[last] = dht,   dH_end[p] = diag(D_{p+1}) dH_end[p+1] + Lr_{p+1}.
// The consumers fold these recurrences over the earlier (later) pieces of
// their document when they start (piece_state_in / piece_grad_out in
// tc.cuh); the local states come from piece_state_kernel below.  This file
// also builds the unit table and the launch order of packed documents and
// sizes the workspace.
#include <atomic>

#include "tc_gla_fwd.cuh"

namespace glacore {
namespace tc {

// One CTA: packed documents -> pieces of `plen` tokens, in document order
// (the pieces of one document are consecutive units); units past the last
// piece are empty.
__global__ void __launch_bounds__(1024)
    build_units_kernel(Docs docs, int64_t plen, Unit *units, int64_t max_units) {
  __shared__ int64_t wbuf[32];
  __shared__ int64_t base_of_chunk;
  int64_t off = 0;
  for (int64_t base = 0; base < docs.n; base += blockDim.x) {
    const int64_t d = base + threadIdx.x;
    int64_t np = 0, s = 0, e = 0;
    if (d < docs.n) {
      docs.range(d, s, e);
      np = (e - s + plen - 1) / plen;
    }
    int64_t tot;
    const int64_t ex = block_excl_scan(np, wbuf, tot);
    for (int64_t p = 0; p < np; ++p) {
      const int64_t u = off + ex + p;
      if (u >= max_units) break;
      Unit r;
      r.start = s + p * plen;
      r.end = min(e, r.start + plen);
      r.doc = (int32_t)d;
      r.piece = (int32_t)p;
      r.npieces = (int32_t)np;
      r.pad = 0;
      units[u] = r;
    }
    off += tot;
  }
  if (threadIdx.x == 0) base_of_chunk = off;
  __syncthreads();
  for (int64_t u = base_of_chunk + threadIdx.x; u < max_units; u += blockDim.x) {
    Unit r;
    r.start = r.end = 0;
    r.doc = r.piece = r.pad = 0;
    r.npieces = 1;
    units[u] = r;
  }
}

cudaError_t launch_build_units(const Docs &docs, int64_t plen, Unit *units, int64_t max_units,
                               cudaStream_t st) {
  build_units_kernel<<<1, 1024, 0, st>>>(docs, plen, units, max_units);
  mark_launch("build_units", st);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// The piece passes.  Unrolled over a piece, its local end state is one
// product, L = sum_t diag(exp(sum of g after t in the piece)) k_t v_t^T =
// Khat^T V (and the reverse pass's state gradient at the piece start is
// sum_t diag(exp(sum of g from the piece start to t)) scale q_t do_t^T), so
// each chunk's k (q) is scaled by its decay to the piece end (from the piece
// start) and its product accumulates in TMEM: no per-chunk state step.
// One CTA per (unit, head, key-channel half kb) accumulates
//   L[kb rows]^T = V^T khat[:, kb]      (128 value lanes x 64 channel columns)
// so no CTA needs another's prepared tile.  320 threads, about 100 KB of
// shared memory and 64 TMEM columns: two CTAs share an SM.
//   warp 0     TMA: the kb block of k (q) and all of v (do), 4-stage ring
//   warp 1     TMEM owner and MMA issuer
//   warps 2..9 prep (gates loaded a chunk ahead, prefix / suffix products, the
//              kb block scaled in place), then the store of L and of the
//              piece's total decay of their channels
// ---------------------------------------------------------------------------
namespace psm {
constexpr int NS = 4;
constexpr uint32_t K = 0;         // 4 x 8 KB: the kb column block of k (q), gated in place
constexpr uint32_t V = 32768;     // 4 x 16 KB: v (do), 128 columns
constexpr uint32_t XCH = 98304;   // 2 x 8 x 128 fp32 eighth-chunk gate products
constexpr uint32_t BYTES = 106496;
}  // namespace psm

// bx: CTA index of the pass (2 per unit).  With uniform rows (implicit
// units, npr pieces per row) only the units that contribute are launched:
// CTA pair w is piece w % (npr - 1) (+1 for the reverse pass) of row
// w / (npr - 1); with a unit table (npr = 0) every unit is launched and the
// ones with nothing to contribute exit.
template <bool REV>
__device__ __forceinline__ void piece_state_body(const FwdMaps &maps, const FwdArgs &a, unsigned bx, int npr) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t full[psm::NS], empty[psm::NS], prep_done[psm::NS], u_done;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = bx & 1, h = blockIdx.y;
  const int64_t w = bx >> 1;
  const int64_t u = npr > 1 ? (w / (npr - 1)) * npr + w % (npr - 1) + (REV ? 1 : 0) : w;
  const Unit un = a.units.get(u);
  const int64_t s0 = un.start, s1 = un.end;
  // the forward pass has nothing to hand on from a document's last piece,
  // the reverse pass nothing from its first
  if (!a.all_units && (REV ? un.piece == 0 : un.piece == un.npieces - 1)) return;
  const int nch = (int)((s1 - s0 + C - 1) / C);
  if (nch <= 0) return;
  // forward pass: chunks last to first (decay to the piece end); reverse: first to last
  auto chunk_tok = [&](int j) -> int64_t { return s0 + (int64_t)(REV ? j : nch - 1 - j) * C; };

  if (warp == 1) {
    tmem_alloc(&tmem_base, 64);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < psm::NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&prep_done[i], 256);
    }
    mbar_init(&u_done, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t sbase = smem_u32(sm);
  volatile int *abortp = &abort_flag;
#define PS_FAIL_AND_BREAK       \
  {                             \
    atomicExch(&abort_flag, 1); \
    break;                      \
  }

  if (warp == 0) {
    if (lane == 0) {
      const int hq = a.hq_div > 1 ? h / a.hq_div : h;  // head of the k slot's tensor (k or q)
      tma_prefetch_desc(&maps.k);
      tma_prefetch_desc(&maps.v);
      if (!a.gate_head) tma_prefetch_desc(&maps.g);
      for (int j = 0; j < nch; ++j) {
        const int s = j % psm::NS;
        if (j >= psm::NS && !mbar_wait(&empty[s], ((j / psm::NS) - 1) & 1, WAIT_CYCLES)) PS_FAIL_AND_BREAK
        if (*abortp) break;
        const int tok = (int)chunk_tok(j);
        mbar_expect_tx(&full[s], 8192 + 16384);
        tma_load_3d(sm + psm::K + s * 8192, &maps.k, 64 * kb, hq, tok, &full[s]);
        tma_load_3d(sm + psm::V + s * 16384, &maps.v, 0, h, tok, &full[s]);
        tma_load_3d(sm + psm::V + s * 16384 + 8192, &maps.v, 64, h, tok, &full[s]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idU = idesc_bf16(128, 64, true, true);
      uint32_t ph = 0;
      for (int j = 0; j < nch; ++j) {
        const int s = j % psm::NS;
        if (!mbar_wait(&prep_done[s], (ph >> s) & 1, WAIT_CYCLES)) PS_FAIL_AND_BREAK
        ph ^= 1u << s;
        tc_fence_after();
        const uint32_t ka = sbase + psm::K + s * 8192, va = sbase + psm::V + s * 16384;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tbase, mdesc(va, ks, 8192), mdesc(ka, ks, 8192), idU, (j > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&empty[s]);
        if (j == nch - 1) mma_commit(&u_done);
      }
      // the last commits have landed before the CTA leaves
      for (int j = max(0, nch - psm::NS); j < nch && !*abortp; ++j)
        if (!mbar_wait(&empty[j % psm::NS], (j / psm::NS) & 1, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
    }
  } else {
    // prep warps: channels c0, c0 + 1 of this CTA's half, tokens 8 pw .. 8 pw + 7
    const int pw = warp - 2;
    const int c0 = 64 * kb + 2 * lane, t0 = 8 * pw;
    uint32_t ph_full = 0;
    float2 dec = make_float2(1.f, 1.f);  // decay of the channels over the visited chunks
    float2 xn[8];
    auto load_x = [&](int jj, float2 (&x)[8]) {
      const int64_t tk = chunk_tok(jj);
      const int LL = (int)min((int64_t)C, s1 - tk);
      if (a.gate_head) {  // one gate per head: the same for both channels
        const float *gp = a.g + (tk + t0) * a.H + h;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float gv = (t0 + i < LL) ? ldg_early(gp + (int64_t)i * a.H) : 0.f;
          x[i] = make_float2(gv, gv);
        }
      } else {
        const float *gp = a.g + ((tk + t0) * a.H + h) * KD + c0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          x[i] = (t0 + i < LL) ? ldg_early2(gp + (int64_t)i * a.H * KD) : make_float2(0.f, 0.f);
      }
    };
    load_x(0, xn);
    for (int j = 0; j < nch; ++j) {
      const int s = j % psm::NS;
      const int L = (int)min((int64_t)C, s1 - chunk_tok(j));
      float2 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = xn[i];
      if (j + 1 < nch) load_x(j + 1, xn);
      // on a failed wait the warps still pass the named barrier inside the
      // prep (all eight must), with the abort recorded
      if (!mbar_wait(&full[s], (ph_full >> s) & 1, WAIT_CYCLES)) atomicExch(&abort_flag, 1);
      ph_full ^= 1u << s;
      // the kb block sits in an 8 KB slot: pass the tile base one block lower for kb = 1
      const uint32_t kt = sbase + psm::K + s * 8192 - (uint32_t)kb * 8192u;
      const float2 tot = prep_chunk_pair(kt, kt, x, nullptr, reinterpret_cast<float *>(sm + psm::XCH) + (j & 1) * 1024,
                                         pw, lane, kb, L, a.scale, false, REV, true, dec);
      dec.x *= tot.x;
      dec.y *= tot.y;
      fence_async_smem();
      mbar_arrive(&prep_done[s]);
    }
    if (pw == 0 && !*abortp) {
      a.dbuf[(u * a.H + h) * KD + c0] = dec.x;
      a.dbuf[(u * a.H + h) * KD + c0 + 1] = dec.y;
    }
    // L^T in TMEM: lane = value column v, column = channel 64 kb + col.  Warps
    // of the same lane quarter split the 64 columns.
    const int v = 32 * (warp & 3) + lane, half = (warp - 2) >> 2;
    const bool done = mbar_wait(&u_done, 0, WAIT_CYCLES);
    __syncwarp();
    if (done) {
      tc_fence_after();
      uint32_t r[16], r2[16];
      const uint32_t ta = tbase + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * half;
      tmem_ld16(ta, r);
      tmem_ld16(ta + 16, r2);
      tmem_ld_wait(r);
      tmem_tie(r2);
      if (!*abortp) {
        float *dst = a.lbuf + ((u * a.H + h) * KD + 64 * kb + 32 * half) * VD + v;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          dst[(int64_t)i * VD] = __uint_as_float(r[i]);
          dst[(int64_t)(16 + i) * VD] = __uint_as_float(r2[i]);
        }
      }
    } else {
      atomicExch(&abort_flag, 1);
    }
  }
#undef PS_FAIL_AND_BREAK
  tc_fence_before();
  __syncthreads();
  if (*abortp && threadIdx.x == 0) set_device_error(a.err, GLACORE_ERR_TIMEOUT);
  if (warp == 1) tmem_dealloc(tbase, 64);
}

// CTAs x < nfwd: forward piece pass (key half x % 2); the rest the reverse
// piece pass (x - nfwd likewise).
__global__ void __launch_bounds__(320, 2)
    piece_state_kernel(const __grid_constant__ FwdMaps fm, const FwdArgs fa, const __grid_constant__ FwdMaps rm,
                       const FwdArgs ra, unsigned nfwd, int npr) {
  if (blockIdx.x < nfwd)
    piece_state_body<false>(fm, fa, blockIdx.x, npr);
  else
    piece_state_body<true>(rm, ra, blockIdx.x - nfwd, npr);
}

cudaError_t launch_piece_states(const FwdMaps &fm, const FwdArgs &fa, const FwdMaps *rm, const FwdArgs *ra,
                                int64_t units, int64_t H, cudaStream_t st, bool rev_only) {
  const int smem = psm::BYTES + 1024;
  cudaError_t e = cudaFuncSetAttribute(piece_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // all of the unified L1 / shared memory as shared memory, so that two CTAs fit on an SM
  e = cudaFuncSetAttribute(piece_state_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  // uniform rows: launch only the npr - 1 contributing pieces of each row
  int npr = 0;
  int64_t work = units;
  if (!fa.units.table && fa.units.plen > 0) {
    npr = (int)((fa.units.docs.T + fa.units.plen - 1) / fa.units.plen);
    work = (units / npr) * (npr - 1);
  }
  if (work <= 0) return cudaSuccess;
  const unsigned nfwd = (unsigned)(2 * work);
  if (rev_only && !rm) return cudaErrorInvalidValue;
  const dim3 grid(rev_only ? nfwd : (rm ? 2 * nfwd : nfwd), (unsigned)H);
  piece_state_kernel<<<grid, 320, smem, st>>>(fm, fa, rm ? *rm : fm, ra ? *ra : fa, rev_only ? 0u : nfwd, npr);
  mark_launch("piece_state_kernel", st);
  return cudaGetLastError();
}

// One CTA: counting sort of the units by chunk count, longest first (ties in
// any order; results do not depend on the launch order).
__global__ void __launch_bounds__(1024) order_units_kernel(Units us, int64_t n, int32_t *order) {
  __shared__ int cnt[1024];
  for (int i = threadIdx.x; i < 1024; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  auto bucket = [&](int64_t u) -> int {
    const Unit un = us.get(u);
    return (int)min((int64_t)1023, (un.end - un.start + C - 1) / C);
  };
  for (int64_t u = threadIdx.x; u < n; u += blockDim.x) atomicAdd(&cnt[bucket(u)], 1);
  __syncthreads();
  {  // cnt[b] <- first position of bucket b (longer buckets first): thread t scans bucket 1023 - t
    __shared__ int64_t wbuf[32];
    const int b = 1023 - (int)threadIdx.x;
    int64_t tot;
    const int64_t pos = block_excl_scan((int64_t)cnt[b], wbuf, tot);
    cnt[b] = (int)pos;
  }
  __syncthreads();
  for (int64_t u = threadIdx.x; u < n; u += blockDim.x) order[atomicAdd(&cnt[bucket(u)], 1)] = (int32_t)u;
}

cudaError_t launch_order_units(const Units &us, int64_t n, int32_t *order, cudaStream_t st) {
  Units plain = us;
  plain.order = nullptr;
  order_units_kernel<<<1, 1024, 0, st>>>(plain, n, order);
  mark_launch("order_units", st);
  return cudaGetLastError();
}

// Piece length: split documents only when (documents x heads x CTAs per
// unit) leaves most of the GPU's SMs idle, and then into about as many
// pieces as make one wave.
// SMs of the current device (one CTA of the chunk-walking kernels per SM).
static int64_t sm_count() {
  static std::atomic<int> cache[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int64_t piece_len(const glacore_problem *p, bool backward) {
  const int64_t sms = sm_count();
  const int64_t per_unit = backward ? 1 : 2;
  const int64_t units = p->n_seqs * p->H * per_unit;
  const int64_t never = (int64_t)1 << 40;
  if (units <= 0 || units * 4 >= sms * 3) return never;
  const int64_t want = sms / units;  // pieces per document
  if (want < 2) return never;
  const int64_t avg = (p->B * p->T + p->n_seqs - 1) / p->n_seqs;
  int64_t plen = (avg + want - 1) / want;
  plen = ((plen + C - 1) / C) * C;
  if (plen < 4 * C) plen = 4 * C;
  return plen >= avg ? never : plen;
}

int64_t max_units_of(const glacore_problem *p, int64_t plen) {
  if (plen >= ((int64_t)1 << 40)) return p->n_seqs;
  if (!p->segment_ids) return p->B * ((p->T + plen - 1) / plen);
  return p->n_seqs + (p->B * p->T + plen - 1) / plen;
}

static size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

TcLayout tc_layout(const glacore_problem *p, bool backward) {
  TcLayout L;
  L.plen = piece_len(p, backward);
  L.pieces = L.plen < ((int64_t)1 << 40);
  L.table = L.pieces && p->segment_ids != nullptr;
  L.max_units = max_units_of(p, L.plen);
  const size_t mu = (size_t)L.max_units, H = (size_t)p->H;
  const size_t state = (size_t)KD * VD * sizeof(float);
  size_t off = 0;
  L.off_units = L.off_order = L.off_L = L.off_D = L.off_Lr = L.off_Dr = L.off_dgp = L.off_bvec = L.off_ckpt = 0;
  L.off_qt = L.off_kt = L.off_eng = L.off_egam = 0;
  // chunks of all documents (upper bound) -> checkpoint slots
  const int64_t chunks = p->segment_ids ? (p->B * p->T + C - 1) / C + p->n_seqs
                                        : p->B * ((p->T + C - 1) / C);
  L.ckpt_slots = chunks / CKPT_CHUNKS + 1;
  if (p->segment_ids) {  // launch order of the units of a packed batch
    L.off_order = off;
    off = al256(off + mu * sizeof(int32_t));
  }
  if (L.pieces) {
    if (L.table) {
      L.off_units = off;
      off = al256(off + mu * sizeof(Unit));
    }
    L.off_L = off;
    off = al256(off + mu * H * state);
    L.off_D = off;
    off = al256(off + mu * H * KD * sizeof(float));
    if (backward) {
      L.off_Lr = off;
      off = al256(off + mu * H * state);
      L.off_Dr = off;
      off = al256(off + mu * H * KD * sizeof(float));
    }
  }
  if (backward) {
    // q (.) dq partials per chunk slot (global chunk index), channel-major
    L.off_dgp = off;
    off = al256(off + (size_t)chunks * H * KD * C * sizeof(float));
    L.off_bvec = off;
    off = al256(off + mu * H * KD * sizeof(float));
    L.off_ckpt = off;
    off = al256(off + (size_t)L.ckpt_slots * H * state);
    // gated operands of pass B, written by pass A: qt = scale q exp(G), kt = k exp(-G)
    L.off_qt = off;
    off = al256(off + (size_t)p->B * p->T * H * KD * 2);
    L.off_kt = off;
    off = al256(off + (size_t)p->B * p->T * H * KD * 2);
    // exp(-G) per chunk slot (pass A -> pass B), bf16, laid out as the partials
    L.off_eng = off;
    off = al256(off + (size_t)chunks * H * KD * C * sizeof(uint16_t));
    // each chunk slot's exp(-Gam), fp32
    L.off_egam = off;
    off = al256(off + (size_t)chunks * H * KD * sizeof(float));
  }
  L.total = off;
  return L;
}

}  // namespace tc
}  // namespace glacore
