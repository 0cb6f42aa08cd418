// tc_common.cuh -- helpers shared by the tcgen05 GLA kernels (tensor maps,
// operand descriptors, packed bf16 shared/global stores, swizzled row
// addressing).  K = V = 128, chunk C = 64.
#pragma once

#include "tc.cuh"
#include "tc_ptx.cuh"

namespace glacore {
namespace tc {

using namespace ptx;

constexpr long long WAIT_CYCLES = 4000000000LL;  // ~2 s: bounded waits

// Smallest total decay exp(sum of g over a chunk) of one channel that the
// chunk-local factorisation exp(G_t) * exp(-G_s) keeps inside the fp32 /
// bf16 exponent range: exp(-80).  A chunk below it makes the kernel record
// GLACORE_ERR_RANGE (its outputs are then not valid).
constexpr float kMinChunkDecay = 1.8048513e-35f;

typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                             const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                             const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                             CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Makes the current device's primary context current in this host thread.
// The tensor maps are encoded through the driver API, which needs a current
// context; the runtime binds one only when a runtime call needs it, so a
// host thread that has made no CUDA call yet would have none.
inline cudaError_t bind_context() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaSetDevice(dev);
  return e;
}

inline EncodeFn encoder() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeFn)p;
  }
  return fn;
}

// 3-D map over a [BT, heads, D] tensor: dims (D, heads, BT), box
// (box_x, 1, C tokens), 128-byte swizzle (box_x = 64 bf16 or 32 fp32
// elements: one 128-byte row per token).  row_stride: elements between
// consecutive tokens (0: heads * D, contiguous).
inline bool make_map(CUtensorMap *m, const void *base, bool bf16, int64_t D, int64_t heads,
                     int64_t BT, int box_x, int64_t row_stride = 0, int box_rows = C) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  const int es = bf16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)BT};
  cuuint64_t strides[2] = {(cuuint64_t)(D * es), (cuuint64_t)((row_stride ? row_stride : heads * D) * es)};
  cuuint32_t box[3] = {(cuuint32_t)box_x, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                   const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_global_v4(void *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
// Read-only global loads issued where they stand: a volatile asm keeps the
// compiler from sinking them to their first use, so loads meant for the next
// chunk stay in flight while the current one is processed.
__device__ __forceinline__ float ldg_early(const float *p) {
  float r;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ float2 ldg_early2(const float *p) {
  float2 r;
  asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(r.x), "=f"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
__device__ __forceinline__ float4 ldg_early4(const float *p) {
  float4 r;
  asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p));
  return r;
}
__device__ __forceinline__ float bf16_at(const uint8_t *tile, uint32_t off) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + off));
}
__device__ __forceinline__ void put_bf16(uint8_t *tile, uint32_t off, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(tile + off) = __float2bfloat16_rn(x);
}

// K-major descriptor step ks (16 elements along K) of a tile whose K extent
// is split into 64-element column blocks of `rows` rows each.
__device__ __forceinline__ SDesc kdesc(uint32_t base, int ks, uint32_t rows) {
  return sdesc_sw128(base, 16, 1024) + ((uint32_t)(ks >> 2) * rows * 128u + (uint32_t)(ks & 3) * 32u);
}
// MN-major descriptor step ks (16 rows along K) of a tile of K rows whose
// M/N extent is split into 64-element column blocks `blk` bytes apart.
__device__ __forceinline__ SDesc mdesc(uint32_t base, int ks, uint32_t blk) {
  return sdesc_sw128(base, blk, 1024) + (uint32_t)ks * 2048u;
}


// Per-thread TMEM helpers for 32-column blocks (32x32b shape, .x32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait32(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Shared-memory addresses of one column c of a tile with the 128-byte
// swizzle, rows r0 + i (r0 % 8 == 0): the XOR pattern depends only on the
// row mod 8, so eight bases cover every row and the row term of at(i)
// folds into the instruction's immediate once loops are unrolled.
//   ColBf16: bf16 tile of 64-column blocks, 64 rows each (TMA box 64 x 64)
//   ColF32:  fp32 tile of 32-column blocks, 64 rows each (TMA box 32 x 64)
struct ColBf16 {
  uint32_t a[8];
  // blk: distance between the tile's two 64-column blocks
  __device__ __forceinline__ ColBf16(uint32_t tile, int r0, int c, uint32_t blk = 8192u) {
    const uint32_t b = tile + (uint32_t)(c >> 6) * blk + (uint32_t)r0 * 128u + (uint32_t)(c & 7) * 2u;
    const uint32_t cc = (uint32_t)(c >> 3) & 7u;
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = b + ((cc ^ (uint32_t)k) << 4);
  }
  __device__ __forceinline__ uint32_t at(int i) const { return a[i & 7] + (uint32_t)i * 128u; }
};
struct ColF32 {
  uint32_t a[8];
  __device__ __forceinline__ ColF32(uint32_t tile, int r0, int c) {
    const uint32_t b = tile + (uint32_t)(c >> 5) * 8192u + (uint32_t)r0 * 128u + (uint32_t)(c & 3) * 4u;
    const uint32_t cc = (uint32_t)(c >> 2) & 7u;
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = b + ((cc ^ (uint32_t)k) << 4);
  }
  __device__ __forceinline__ uint32_t at(int i) const { return a[i & 7] + (uint32_t)i * 128u; }
};
__device__ __forceinline__ uint16_t lds_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v));
}
__device__ __forceinline__ float lds_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v));
}

// Plain (compiler-visible) 16-bit shared accesses through a generic pointer,
// so that independent loads can be batched and scheduled early.
__device__ __forceinline__ uint16_t ld_u16(const uint8_t *p) {
  return *reinterpret_cast<const uint16_t *>(p);
}
__device__ __forceinline__ void st_u16(uint8_t *p, uint16_t v) { *reinterpret_cast<uint16_t *>(p) = v; }
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t *>(&h);
}

// In-register 4 x 4 transposes across groups of 4 lanes.  On entry lane l
// holds v[t] = value of channel (its own) at token t (t = 0..15).  On exit
// v[4 s + e] = value of channel 4 (l / 4) + e (of the warp's 32) at token
// 4 s + (l % 4): each lane then owns 4 consecutive channels of one token, so
// the epilogue can store 8 or 16 contiguous bytes instead of one element.
// Butterfly over lane bits 1 and 0 (shfl_xor 2, then 1).
__device__ __forceinline__ void transpose_4x4_blocks(float (&v)[16], int lane) {
  const bool b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float send = b1 ? v[4 * s + j] : v[4 * s + j + 2];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 2);
      if (b1)
        v[4 * s + j] = recv;
      else
        v[4 * s + j + 2] = recv;
    }
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const float send = b0 ? v[4 * s + j] : v[4 * s + j + 1];
      const float recv = __shfl_xor_sync(0xffffffffu, send, 1);
      if (b0)
        v[4 * s + j] = recv;
      else
        v[4 * s + j + 1] = recv;
    }
  }
}

// Stores 16 tokens x 32 channels held as after transpose_4x4_blocks:
// `row0` points at (token t_base, channel c_base of the warp), rows `stride`
// elements apart; rows t_base + t >= L are skipped.
__device__ __forceinline__ void store_block_f32(float *row0, int64_t stride, const float (&v)[16],
                                                int lane, int t_in_chunk0, int L) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int t = 4 * s + (lane & 3);
    if (t_in_chunk0 + t < L)
      *reinterpret_cast<float4 *>(row0 + (int64_t)t * stride + 4 * (lane >> 2)) =
          make_float4(v[4 * s], v[4 * s + 1], v[4 * s + 2], v[4 * s + 3]);
  }
}
// cmax: the block's columns at or past cmax are skipped.
__device__ __forceinline__ void store_block_bf16(__nv_bfloat16 *row0, int64_t stride, const float (&v)[16],
                                                 int lane, int t_in_chunk0, int L, int cmax = 32) {
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int t = 4 * s + (lane & 3);
    if (t_in_chunk0 + t < L && 4 * (lane >> 2) < cmax) {
      uint2 w;
      w.x = pack_bf16(v[4 * s], v[4 * s + 1]);
      w.y = pack_bf16(v[4 * s + 2], v[4 * s + 3]);
      *reinterpret_cast<uint2 *>(row0 + (int64_t)t * stride + 4 * (lane >> 2)) = w;
    }
  }
}

// Orders the uses of registers filled by an earlier tcgen05.ld after a
// tcgen05.wait::ld that was tied to other registers (volatile asm statements
// keep their order): lets one wait cover several loads.
__device__ __forceinline__ void tmem_tie(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}

// Masked C x C tiles (causal mask col <= row) in shared memory: bf16
// K-major [row][col] with the 128-byte swizzle, written from an fp32
// accumulator in the M = 64 TMEM layout (row r in lane 32 (r / 16) + r % 16).
// Warp quarter qw owns rows 16 qw .. 16 qw + 15, so its 16-column blocks
// cb > qw are zero for every chunk: mask_tile_init writes them once, and
// mask_tile_to_smem then loads and writes only the blocks cb <= qw (the
// diagonal block cb == qw with the mask).  Nothing else may write the tile.
__device__ __forceinline__ void mask_block_store(uint8_t *tile, int row, int cb, const uint32_t (&r)[16],
                                                 bool diag, int lane) {
#pragma unroll
  for (int hb = 0; hb < 2; ++hb) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i0 = hb * 8 + 2 * e;
      const float x0 = (!diag || i0 <= lane) ? __uint_as_float(r[i0]) : 0.f;
      const float x1 = (!diag || i0 + 1 <= lane) ? __uint_as_float(r[i0 + 1]) : 0.f;
      w[e] = pack_bf16(x0, x1);
    }
    st_shared_v4(smem_u32(tile + sw128_off(row, cb * 16 + hb * 8, 64)), w[0], w[1], w[2], w[3]);
  }
}
__device__ __forceinline__ void mask_tile_init(uint8_t *tile, int qw, int lane) {
  if (lane < 16) {
    const int row = qw * 16 + lane;
    for (int cb = qw + 1; cb < 4; ++cb)
#pragma unroll
      for (int hb = 0; hb < 2; ++hb)
        st_shared_v4(smem_u32(tile + sw128_off(row, cb * 16 + hb * 8, 64)), 0u, 0u, 0u, 0u);
  }
}
// The same tile from an M = 128 accumulator (row r in lane r): the warp of
// one TMEM lane quarter writes rows r0 .. r0 + 31 (r0 = 0 or 32; t_acc
// addresses the tile's first column in that quarter).  mask_rows_init writes
// each row's zero blocks above the diagonal once; mask_rows_to_smem loads
// the blocks up to the warp's last diagonal block and writes, per row, the
// blocks at or below its diagonal (diagonal block masked).
__device__ __forceinline__ void mask_rows_init(uint8_t *tile, int r0, int lane) {
  const int row = r0 + lane;
  for (int cb = (row >> 4) + 1; cb < 4; ++cb)
#pragma unroll
    for (int hb = 0; hb < 2; ++hb)
      st_shared_v4(smem_u32(tile + sw128_off(row, cb * 16 + hb * 8, 64)), 0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void mask_rows_to_smem(uint32_t t_acc, int r0, int lane, uint8_t *tile) {
  const int row = r0 + lane, rb = row >> 4;
#pragma unroll
  for (int cp = 0; cp < 4; cp += 2) {
    if (cp <= (r0 >> 4) + 1) {
      uint32_t a0[16], a1[16];
      tmem_ld16(t_acc + cp * 16, a0);
      tmem_ld16(t_acc + cp * 16 + 16, a1);
      tmem_ld_wait(a0);
      tmem_tie(a1);
      if (cp <= rb) mask_block_store(tile, row, cp, a0, cp == rb, row & 15);
      if (cp + 1 <= rb) mask_block_store(tile, row, cp + 1, a1, cp + 1 == rb, row & 15);
    }
  }
}
// The masked tile as two bf16 tiles, hi = bf16(x) and lo = bf16(x - hi):
// hi + lo carries about 16 bits of the fp32 value, so a product with both
// (two accumulating MMAs) removes the bf16 rounding of the tile itself.
__device__ __forceinline__ void mask_block_store_hilo(uint8_t *hi_tile, uint8_t *lo_tile, int row, int cb,
                                                      const uint32_t (&r)[16], bool diag, int rl) {
#pragma unroll
  for (int hb = 0; hb < 2; ++hb) {
    uint32_t w[4], wl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i0 = hb * 8 + 2 * e;
      const float x0 = (!diag || i0 <= rl) ? __uint_as_float(r[i0]) : 0.f;
      const float x1 = (!diag || i0 + 1 <= rl) ? __uint_as_float(r[i0 + 1]) : 0.f;
      w[e] = pack_bf16(x0, x1);
      wl[e] = pack_bf16(x0 - __uint_as_float(w[e] << 16), x1 - __uint_as_float(w[e] & 0xffff0000u));
    }
    const uint32_t off = sw128_off(row, cb * 16 + hb * 8, 64);
    st_shared_v4(smem_u32(hi_tile + off), w[0], w[1], w[2], w[3]);
    st_shared_v4(smem_u32(lo_tile + off), wl[0], wl[1], wl[2], wl[3]);
  }
}
// mask_tile_to_smem into a hi / lo pair of tiles (both set up by
// mask_tile_init).  The M = 64 accumulator holds a warp's 16 rows in lanes
// 0..15; lanes 16..31 take the second 16-column block of each pair, shuffled
// over from lanes 0..15, so every lane writes one block (hi and lo).
__device__ __forceinline__ void mask_tile_to_smem_hilo(uint32_t t_acc, uint32_t lane_off, int qw, int lane,
                                                       uint8_t *hi_tile, uint8_t *lo_tile) {
  const int rl = lane & 15, row = qw * 16 + rl;
  const bool second = lane >= 16;
#pragma unroll
  for (int cp = 0; cp < 4; cp += 2) {
    if (cp <= qw) {
      uint32_t r0[16], r1[16];
      tmem_ld16(t_acc + lane_off + cp * 16, r0);
      tmem_ld16(t_acc + lane_off + cp * 16 + 16, r1);
      tmem_ld_wait(r0);
      tmem_tie(r1);
      uint32_t v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t s = __shfl_sync(0xffffffffu, r1[i], rl);
        v[i] = second ? s : r0[i];
      }
      const int cb = cp + (second ? 1 : 0);
      if (cb <= qw) mask_block_store_hilo(hi_tile, lo_tile, row, cb, v, cb == qw, rl);
    }
  }
}
// Called by a whole warp of the epilogue warpgroup (warp quarter qw).
__device__ __forceinline__ void mask_tile_to_smem(uint32_t t_acc, uint32_t lane_off, int qw, int lane,
                                                  uint8_t *tile) {
  const int row = qw * 16 + lane;
#pragma unroll
  for (int cp = 0; cp < 4; cp += 2) {
    if (cp <= qw) {
      uint32_t r0[16], r1[16];
      tmem_ld16(t_acc + lane_off + cp * 16, r0);
      tmem_ld16(t_acc + lane_off + cp * 16 + 16, r1);
      tmem_ld_wait(r0);
      tmem_tie(r1);
      if (lane < 16) {
        mask_block_store(tile, row, cp, r0, cp == qw, lane);
        if (cp + 1 <= qw) mask_block_store(tile, row, cp + 1, r1, cp + 1 == qw, lane);
      }
    }
  }
}

}  // namespace tc
}  // namespace glacore
