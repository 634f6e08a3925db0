// Bulk quantize of d = 128 bf16 vectors with the products on tensor cores.
//
// [Reconstruction] §5 Steps 1-5 and §6; [Design study] §CPU and WASM kernel
// design ("Append-time key kernel") and §Packed format.  Same results as
// quantize_tile (every decision on fp32 values of the same accuracy), laid
// out for mma.m16n8k16:
//
//   * one warp owns a tile of 16 vectors (the M rows of the MMAs) of one kv
//     head; coordinates are permuted inside each 16-wide k-block so that one
//     16-byte load per lane yields two A fragments, and so that every lane
//     holds 4 consecutive coordinates per block of the outputs: a lane owns
//     one byte of every packed 32-bit word (a byte transpose across the quad
//     assembles the words);
//   * FWHT: H_128 = H_8 (x) H_16 over a split of the 7 index bits; the
//     H_16 factor (with the sign flips folded in) is one bf16 MMA per
//     k-block (+-1 and bf16 inputs are exact, accumulation in fp32), the
//     H_8 factor a register butterfly across the 8 accumulator blocks;
//   * dense Pi: bf16 inputs against Pi split in three bf16 limbs (24
//     significant bits), fragments staged once per CTA in shared memory;
//   * codes: sign and magnitude, the magnitude by binary search over the
//     positive boundaries held in registers (bit width a template
//     parameter); planes packed four at a time with one multiply;
//   * QJL keys (quantize_keys_tc_kernel): a CTA of 8 warps holds 128
//     vectors, one UMMA M = 128 tile; S r runs as tcgen05.mma over hi / lo
//     f16 limbs of r and S (hi*hi + hi*lo + lo*hi) into tensor memory (the
//     structured S = H diag(sigma_S) is synthesised from its signs: exact
//     +-1 limbs).
//     Every entry whose magnitude is below a certified bound of the limb and
//     accumulation errors (6e-5 ||r|| ||S_c||, a few per thousand vectors)
//     is recomputed in fp32 by the warp from the limbs, so every sign is
//     that of the fp32 product up to 2^-21 relative;
//   * norms in fp32 with balanced summation trees (relative error at most
//     about 8 u before the square root halves it), scales taken as
//     sqrt(d / s) and sqrt(s_r / d) (d a power of two).
//
// Requirements checked by the launcher: d = 128, bf16 input, 16-byte aligned
// input, codebook tables antisymmetric (c[half+m] = -c[half-1-m], middle
// boundary 0, increasing boundaries).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <limits.h>
#include <math.h>
#include <string.h>

#include "tq_device.cuh"

namespace tq {

// The including file defines tq::g_quant_err (the device error word of the
// quantize / append kernels) before including this header.

namespace wq {

constexpr int D = 128;
constexpr int KB = D / 16;     // k-blocks
// code cell tables (see code_cell): 2^(5 + J) + 1 cells of 8 bytes, then 16 records
constexpr int kLutMaxJ = 4;
__host__ __device__ constexpr size_t lut_cells_bytes(int J) { return ((size_t)(32 << J) + 1) * 8; }
// spread: a second cell table for code-only lookups (see code_spread)
__host__ __device__ constexpr size_t lut_bytes(int J, bool spread) {
  return lut_cells_bytes(J) + 16 * 8 + (spread ? lut_cells_bytes(J) : 0);
}

// Permuted coordinates.  Logical index L in [0, 16) of k-block kk sits at
// blk_base(kk) + free_off(L): bits 2, 5, 6 of the coordinate come from the
// block, bits 0, 1, 3, 4 from L.
__host__ __device__ constexpr int blk_base(int kk) { return 32 * (kk >> 1) + 4 * (kk & 1); }
__host__ __device__ constexpr int free_off(int L) { return 8 * ((L >> 1) & 3) + 2 * (L >> 3) + (L & 1); }
// output coordinate of column n in rotation tile nt (tiles 2a', 2a'+1 form block a')
__host__ __device__ constexpr int rot_out(int nt, int n) {
  return blk_base(nt >> 1) + 8 * (n >> 1) + 2 * (nt & 1) + (n & 1);
}
// sketch coordinate of column n in tile nt: tiles 4w..4w+3 cover word w
__host__ __device__ constexpr int sk_out(int nt, int n) {
  return 32 * (nt >> 2) + 8 * (n >> 1) + 2 * (nt & 3) + (n & 1);
}

struct Shared {
  uint2 hfrag[KB][2][32];      // FWHT H_16 * sigma fragments (bf16)
};
constexpr size_t kPfragBytes = (size_t)3 * 16 * KB * 32 * sizeof(uint2);  // Pi limbs (bf16)
// Per-warp block buffer: [2][KB][32] uint4, FWHT only: the rotated tile
// (R = 0 rows in half 0, R = 1 rows in half 1).
constexpr size_t kBlkBytes = (size_t)2 * KB * 32 * sizeof(uint4);

// FWHT: 12 warps, next tile staged in shared memory by cp.async; dense: 8
// warps, two CTAs per SM, next tile prefetched into registers.
__host__ __device__ constexpr int warps_for(bool dense) { return dense ? 8 : 12; }
__host__ __device__ constexpr int ctas_for(bool dense) { return dense ? 2 : 1; }
__host__ __device__ constexpr size_t blk_bytes(bool dense) { return dense ? 0 : (size_t)warps_for(dense) * kBlkBytes; }
__host__ __device__ constexpr size_t stage_bytes(bool dense) {
  return dense ? 0 : (size_t)warps_for(dense) * 8 * 32 * sizeof(uint4);
}

__host__ __device__ constexpr size_t smem_bytes(bool dense) {
  return sizeof(Shared) + (dense ? kPfragBytes : 0) + blk_bytes(dense) + stage_bytes(dense);
}

// 16-byte global -> shared copy; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint32_t bf16_bits(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
__device__ __forceinline__ uint32_t f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Byte transpose across the 4 lanes t of a quad: byte k of v on lane t is
// element (t, k); the result's byte s on lane t is element (s, t).
__device__ __forceinline__ uint32_t quad_transpose(uint32_t v, int t) {
  const uint32_t p = __shfl_xor_sync(0xffffffffu, v, 1);
  const uint32_t a = (t & 1) ? p : v;
  const uint32_t b = (t & 1) ? v : p;
  const uint32_t k0 = t & 1;
  const uint32_t u = __byte_perm(a, b, k0 | ((4 + k0) << 4) | ((k0 + 2) << 8) | ((6 + k0) << 12));
  const uint32_t o = __shfl_xor_sync(0xffffffffu, u, 2);
  return (t < 2) ? __byte_perm(u, o, 0x5410) : __byte_perm(o, u, 0x7632);
}

// Code search by a cell table ([Reconstruction] §5 Step 3: the code of z is
// the number of boundaries t_k <= z, ties up).  The real line is cut into
// cells by
//   cell(z) = RN( sat(RN(z / 32 + 1/2)) * 2^(5 + J) ),
// two fp32 fmas with exact power-of-two scalings, so cell() is monotone and
// the same on the host and the device; J is the smallest scale for which no
// two boundaries share a cell (chosen by the launcher).  Entry i of the cell
// table holds the one boundary b_i in cell i (NaN if none) and the number
// base_i of boundaries in lower cells, so code(z) = base_i + [z >= b_i]
// exactly.  Record c holds centroid c and the sign-magnitude code of c with
// plane p moved to bit 8 p ("spread"), ready to be shifted into a packed word.
// Per coordinate: three fmas, two shared loads, one compare.

__host__ __device__ inline int code_cell(float z, float sc) {
#ifdef __CUDA_ARCH__
  const float s = __saturatef(__fmaf_rn(z, 0.03125f, 0.5f));
  return __float_as_int(__fmaf_rn(s, sc, 12582912.0f)) - 0x4B400000;
#else
  float s = fmaf(z, 0.03125f, 0.5f);
  s = s < 0.f ? 0.f : (s > 1.f ? 1.f : s);
  const float c = fmaf(s, sc, 12582912.0f);
  int bits;
  memcpy(&bits, &c, sizeof bits);
  return bits - 0x4B400000;
#endif
}

// Sign-magnitude code of natural index c of a 2^bits-level antisymmetric book
// (bit 0: z >= 0, bits 1..: number of boundaries between z and 0), spread.
__host__ __device__ constexpr uint32_t spread_code(int c, int bits) {
  return (((c >= (1 << (bits - 1))) ? (1u | ((uint32_t)(c - (1 << (bits - 1))) << 1))
                                    : ((uint32_t)((1 << (bits - 1)) - 1 - c) << 1)) *
          0x204081u) & 0x01010101u;
}

struct CodeLut {
  uint32_t cells;   // shared address of the cell table minus 8 * bits(2^23 + 2^22): cell i at cells + 8 bits(fma)
  uint32_t scells;  // the same for the code-only cell table
  float sc;         // 2^(5 + J)
};

// Builds the tables (all threads of the CTA; a barrier must follow).  bnd:
// the 2^BITS - 1 ascending boundaries, cent: the 2^BITS centroids.  Cell i:
// {b_i, shared address of record base_i}; record c: {centroid c, spread code};
// code-only cell i (SPREAD): {b_i, spread(base_i) | spread(base_i + 1) << 1}.
template <bool SPREAD>
__device__ void build_code_lut_n(unsigned char* at, int J, const float* bnd, const float* cent, int bits, int tid,
                                 int nt) {
  const int NB = (1 << bits) - 1;
  const int BITS = bits;
  float2* cells = reinterpret_cast<float2*>(at);
  uint2* recs = reinterpret_cast<uint2*>(at + lut_cells_bytes(J));
  float2* scells = reinterpret_cast<float2*>(at + lut_cells_bytes(J) + 16 * 8);
  const int nc = (32 << J) + 1;
  const float sc = (float)(32 << J);
  for (int i = tid; i < nc; i += nt) {
    int base = 0, in_cell = 0;
    float b = __int_as_float(0x7fc00000);  // no boundary: NaN, so z >= b is false for every z
    for (int k = 0; k < NB; ++k) {
      const int ck = code_cell(bnd[k], sc);
      base += ck < i ? 1 : 0;
      if (ck == i) {  // one boundary per cell (the launcher's choice of J)
        b = bnd[k];
        ++in_cell;
      }
    }
    if (in_cell > 1) atomicOr(&g_quant_err, TQ_DEVERR_CODEBOOK);
    cells[i] = make_float2(b, __uint_as_float((uint32_t)__cvta_generic_to_shared(recs + base)));
    if (SPREAD)
      scells[i] = make_float2(b, __uint_as_float(spread_code(base, BITS) | (spread_code(min(base + 1, NB), BITS) << 1)));
  }
  for (int c = tid; c <= NB; c += nt) recs[c] = make_uint2(__float_as_uint(cent[c]), spread_code(c, BITS));
}
template <int BITS, bool SPREAD>
__device__ void build_code_lut(unsigned char* at, int J, const float* bnd, const float* cent, int tid, int nt) {
  build_code_lut_n<SPREAD>(at, J, bnd, cent, BITS, tid, nt);
}

__device__ __forceinline__ CodeLut code_lut_at(const unsigned char* at, int J) {
  const uint32_t c = (uint32_t)__cvta_generic_to_shared(at) - 8u * 0x4B400000u;
  return CodeLut{c, c + (uint32_t)(lut_cells_bytes(J) + 16 * 8), (float)(32 << J)};
}

// Shared address of the record of z's code: cell entry, one exact compare
// (z >= b_i: 0 or ~0), record base_i or base_i + 1.
__device__ __forceinline__ uint32_t code_record_addr(float z, const CodeLut& L) {
  const float s = __saturatef(__fmaf_rn(z, 0.03125f, 0.5f));
  const uint32_t cb = __float_as_uint(__fmaf_rn(s, L.sc, 12582912.0f));
  uint32_t ca, ra, ge;
  float b;
  asm("mad.lo.u32 %0, %1, 8, %2;" : "=r"(ca) : "r"(cb), "r"(L.cells));
  asm("ld.shared.v2.b32 {%0, %1}, [%2];" : "=f"(b), "=r"(ra) : "r"(ca));
  asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(ge) : "f"(z), "f"(b));
  return ra - 8u * ge;  // ge = ~0: the next record
}
// Record of the code of z: .x centroid bits, .y spread code.
__device__ __forceinline__ uint2 code_record(float z, const CodeLut& L) {
  uint2 r;
  asm("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(code_record_addr(z, L)));
  return r;
}
// Spread code of z only, from the code-only cell table: one shared load, one compare.
__device__ __forceinline__ uint32_t code_spread(float z, const CodeLut& L) {
  const float s = __saturatef(__fmaf_rn(z, 0.03125f, 0.5f));
  const uint32_t cb = __float_as_uint(__fmaf_rn(s, L.sc, 12582912.0f));
  uint32_t ca, w, ge;
  float b;
  asm("mad.lo.u32 %0, %1, 8, %2;" : "=r"(ca) : "r"(cb), "r"(L.scells));
  asm("ld.shared.v2.b32 {%0, %1}, [%2];" : "=f"(b), "=r"(w) : "r"(ca));
  asm("set.ge.u32.f32 %0, %1, %2;" : "=r"(ge) : "f"(z), "f"(b));
  return (w >> (ge & 1u)) & 0x01010101u;
}

__device__ __forceinline__ float f16lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// Where the records go: flat arrays (bulk quantize) or the page slot of each
// sequence's next token (decode-step append without a window: rows are the
// sequences, the token of sequence b lands in slot seq_len[b] % 16 of page
// block_table[b][seq_len[b] / 16]).
enum { kFlat = 0, kStep = 1 };

// Values, and keys without the QJL sketch (keys with it: quantize_keys_tc_kernel),
// with the key scale where the layer keeps one (EDEN's unbiased scale, which is
// also TurboVec's length-renormalized correction norm / <y, y_hat> once the norm
// is stored on its own: s = 1 / <y, y_hat>).
// DENSE: dense rotation (else FWHT).  grid (x, Hkv).
template <int BITS, bool DENSE, int MODE>
__global__ void __launch_bounds__(32 * warps_for(DENSE), ctas_for(DENSE))
    quantize_warp_kernel(const __grid_constant__ KParams P, const __grid_constant__ KCache C,
                         const __nv_bfloat16* __restrict__ x, long long n_vec, int is_key,
                         uint32_t* __restrict__ codes, uint32_t* __restrict__ signs, float* __restrict__ norms,
                         float* __restrict__ rnorms, int lut_j) {
  constexpr int WARPS = warps_for(DENSE);
  constexpr int NT = 32 * WARPS;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  unsigned char* dyn = smem_raw + sizeof(Shared);
  uint2* pfrag = reinterpret_cast<uint2*>(dyn);  // [3][16][KB][32]
  dyn += DENSE ? kPfragBytes : 0;
  uint4* blk = reinterpret_cast<uint4*>(dyn);    // [WARPS][2][KB][32]
  dyn += blk_bytes(DENSE);
  uint4* stage = reinterpret_cast<uint4*>(dyn);  // [WARPS][8][32]
  dyn += stage_bytes(DENSE);
  unsigned char* lut_at = dyn;                   // code cell table and records

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int head = blockIdx.y;
  const float* ctab = is_key ? P.kc : P.vc;
  const float* ttab = is_key ? P.kt : P.vt;
  const float* rot = (is_key ? P.k_rot : P.v_rot) + (size_t)head * (DENSE ? D * D : D);
  // keys with a scale in place of the sketch (EDEN / length-renormalized, one formula); false otherwise
  const bool corr = is_key && (P.kqjl == TQ_KEY_EDEN || P.kqjl == TQ_KEY_RENORM);
  build_code_lut<BITS, true>(lut_at, lut_j, ttab, ctab, tid, NT);
  const CodeLut lut = code_lut_at(lut_at, lut_j);

  // ---- per-CTA constants.  The four elements of a B fragment (lane (g, t),
  // k-rows 2t, 2t+1, 2t+8, 2t+9 of k-block kk) sit at columns
  // blk_base(kk) + 8t + 0..3 of one row: one aligned float4 per fragment.
  if constexpr (!DENSE) {
    for (int i = tid; i < KB * 2 * 32; i += NT) {
      const int ln = i & 31, nt = (i >> 5) & 1, kk = i >> 6;
      const int gg = ln >> 2, tt = ln & 3;
      const float4 sg = __ldg(reinterpret_cast<const float4*>(rot + blk_base(kk) + 8 * tt));
      const float sv[4] = {sg.x, sg.y, sg.z, sg.w};
      const int out = 8 * (gg >> 1) + 2 * nt + (gg & 1);
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int L = 2 * tt + (e & 1) + 8 * (e >> 1);
        const bool neg = (sv[e] < 0.f) != (bool)(__popc(free_off(L) & out) & 1);
        h[e] = neg ? 0xBF80u : 0x3F80u;
      }
      sh.hfrag[kk][nt][ln] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
  } else {
    constexpr int PER = (16 * KB * 32 + NT - 1) / NT;  // fragments per thread: all loads issued first
    float4 pv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT;
      const int ln = i & 31, kk = (i >> 5) & (KB - 1), nt = (i >> 8) & 15;
      pv[j] = i < 16 * KB * 32
                  ? __ldg(reinterpret_cast<const float4*>(rot + (size_t)rot_out(nt, ln >> 2) * D + blk_base(kk) + 8 * (ln & 3)))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT;
      if (i >= 16 * KB * 32) break;
      const int ln = i & 31, kk = (i >> 5) & (KB - 1), nt = i >> 8;
      const float4 v4 = pv[j];
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      uint32_t l[3][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float l0 = __bfloat162float(__float2bfloat16_rn(v[e]));
        const float l1 = __bfloat162float(__float2bfloat16_rn(v[e] - l0));
        l[0][e] = bf16_bits(v[e]);
        l[1][e] = bf16_bits(v[e] - l0);
        l[2][e] = bf16_bits((v[e] - l0) - l1);
      }
#pragma unroll
      for (int k = 0; k < 3; ++k)
        pfrag[((k * 16 + nt) * KB + kk) * 32 + ln] = make_uint2(l[k][0] | (l[k][1] << 16), l[k][2] | (l[k][3] << 16));
    }
  }
  __syncthreads();

  // ---- tiles of 16 tokens of this head
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 15) / 16;
  const long long stride = (long long)gridDim.x * WARPS;
  uint4* wb = blk + (size_t)warp * 2 * KB * 32;  // this warp's block buffer: wb[(half * KB + a) * 32 + lane]
  auto row_index = [&](long long mt, int R, long long& n) -> bool {
    const long long tok = mt * 16 + g + 8 * R;
    n = tok * P.hkv + head;
    return tok < n_tok && n < n_vec;
  };
  // next tile: registers (dense) or this lane's own slots of the staging area
  uint4 nxt[2][4];  // dense only
  uint4* stg = stage + (size_t)warp * 8 * 32 + lane;  // slot k at stg[32 k]
  auto load = [&](long long mt) {
#pragma unroll
    for (int R = 0; R < 2; ++R) {
      long long n;
      const bool ok = row_index(mt, R, n);
      // row of dh elements, zero-padded to D: 16-byte chunk 4m + t holds coordinates 32m + 8t .. + 7
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(ok ? n : 0) * P.dh) + t;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const bool in = ok && 32 * m + 8 * t < P.dh;
        if constexpr (DENSE) nxt[R][m] = in ? __ldg(src + 4 * m) : make_uint4(0, 0, 0, 0);
        else cp_async16(stg + 32 * (4 * R + m), in ? src + 4 * m : src, in ? 16 : 0);
      }
    }
    if constexpr (!DENSE) cp_async_commit();
  };
  // bulk calls: a CTA's warps take adjacent tiles; a decode-step append spreads its few tiles
  // over CTAs (warp w of CTA c: tile c + gridDim.x w), so each CTA holds one or two
  long long mt = MODE == kStep ? (long long)blockIdx.x + (long long)gridDim.x * warp : (long long)blockIdx.x * WARPS + warp;
  if (mt < n_tiles) load(mt);
  for (; mt < n_tiles; mt += stride) {
    uint4 X[2][4];
    if constexpr (!DENSE) cp_async_wait_all();
#pragma unroll
    for (int R = 0; R < 2; ++R)
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if constexpr (DENSE) X[R][m] = nxt[R][m];
        else X[R][m] = stg[32 * (4 * R + m)];
      }
    if (mt + stride < n_tiles) load(mt + stride);

    long long nrow[2];
    bool okrow[2];
    unsigned char* dst[2] = {nullptr, nullptr};  // step mode: this row's (page, head) sub-block
    int slot[2] = {0, 0};
#pragma unroll
    for (int R = 0; R < 2; ++R) {
      okrow[R] = row_index(mt, R, nrow[R]);
      if constexpr (MODE == kStep) {
        if (okrow[R]) {
          const int b = (int)(nrow[R] / P.hkv);
          const int T = C.seq_len[b];
          const int pidx = T >> 4;
          long long page = -1;
          if (T >= 0 && pidx < C.max_pages) page = C.block_table[(size_t)b * C.max_pages + pidx];
          if (page < 0 || page >= C.n_pages) {
            if (t == 0) atomicOr(&g_quant_err, (T >= 0 && pidx < C.max_pages) ? TQ_DEVERR_PAGE_INDEX : TQ_DEVERR_SEQ_LEN);
            okrow[R] = false;
          } else {
            dst[R] = C.pool + ((size_t)page * P.hkv + head) * (size_t)P.sub_bytes;
            slot[R] = T & 15;
          }
        }
      }
    }

    // norms of rows g (R = 0) and g + 8 (R = 1): squares of bf16 values are
    // exact in fp32; a balanced tree of depth 7 sums them
    float inv[2], nrm[2];
    bool zero[2];
#pragma unroll
    for (int R = 0; R < 2; ++R) {
      float part[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t w[4] = {X[R][m].x, X[R][m].y, X[R][m].z, X[R][m].w};
        float q2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
          q2[k] = lo * lo + hi * hi;
        }
        part[m] = (q2[0] + q2[1]) + (q2[2] + q2[3]);
      }
      float s2 = (part[0] + part[1]) + (part[2] + part[3]);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
      const float n = sqrtf(s2);
      zero[R] = n < kZeroNorm;
      nrm[R] = zero[R] ? 0.f : n;
      // z = sqrt(d) Pi x / n (dense) or H (sigma x) / n (FWHT): one division
      // and one square root of the sum's fp32 value
      inv[R] = zero[R] ? 0.f : sqrtf((DENSE ? (float)D : 1.0f) / s2);
      if (okrow[R] && t == 0) {
        if constexpr (MODE == kFlat) norms[nrow[R]] = nrm[R];
        else reinterpret_cast<float*>(dst[R] + (is_key ? P.off_knorm : P.off_vnorm))[slot[R]] = nrm[R];
      }
    }

    if constexpr (!DENSE) {
      // FWHT: H_16 factor per k-block on tensor cores, H_8 across the blocks,
      // then the rotated tile into the block buffer
      float acc[KB][2][4];
#pragma unroll
      for (int kk = 0; kk < KB; ++kk) {
        const uint4& u0 = X[0][kk >> 1];
        const uint4& u1 = X[1][kk >> 1];
        const uint32_t a0 = (kk & 1) ? u0.z : u0.x, a2 = (kk & 1) ? u0.w : u0.y;
        const uint32_t a1 = (kk & 1) ? u1.z : u1.x, a3 = (kk & 1) ? u1.w : u1.y;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[kk][h][r] = 0.f;
          mma_bf16(acc[kk][h], a0, a1, a2, a3, sh.hfrag[kk][h][lane]);
        }
      }
#pragma unroll
      for (int s = 1; s < KB; s <<= 1)
#pragma unroll
        for (int a = 0; a < KB; ++a)
          if ((a & s) == 0)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const float p = acc[a][h][r], q = acc[a + s][h][r];
                acc[a][h][r] = p + q;
                acc[a + s][h][r] = p - q;
              }
#pragma unroll
      for (int a = 0; a < KB; ++a) {
        wb[(0 * KB + a) * 32 + lane] = make_uint4(__float_as_uint(acc[a][0][0]), __float_as_uint(acc[a][0][1]),
                                                  __float_as_uint(acc[a][1][0]), __float_as_uint(acc[a][1][1]));
        wb[(1 * KB + a) * 32 + lane] = make_uint4(__float_as_uint(acc[a][0][2]), __float_as_uint(acc[a][0][3]),
                                                  __float_as_uint(acc[a][1][2]), __float_as_uint(acc[a][1][3]));
      }
    }

    // codes, two blocks (one packed word) per pass
    uint32_t vword[2][4];      // step mode, values: plane t of words 0..3 of rows g, g + 8
    float ssum[2] = {0.f, 0.f};  // scaled keys: this lane's share of sum |z| c (EDEN) or sum c^2
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      uint32_t Wm[2] = {0u, 0u};  // byte p: plane p of this lane's byte of word m
      float spart[2] = {0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int a = 2 * m + hh;
        float zr[2][4];  // [R][2h + e], before the 1 / n scale
        if constexpr (DENSE) {
          // tiles 2a, 2a+1; the leading limb split over even / odd k-blocks,
          // the small limbs in their own accumulators
          float c[4][2][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int r = 0; r < 4; ++r) c[i][h][r] = 0.f;
#pragma unroll
          for (int kk = 0; kk < KB; ++kk) {
            const uint4& u0 = X[0][kk >> 1];
            const uint4& u1 = X[1][kk >> 1];
            const uint32_t a0 = (kk & 1) ? u0.z : u0.x, a2 = (kk & 1) ? u0.w : u0.y;
            const uint32_t a1 = (kk & 1) ? u1.z : u1.x, a3 = (kk & 1) ? u1.w : u1.y;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint2* pf = pfrag + ((2 * a + h) * KB + kk) * 32 + lane;
              mma_bf16(c[kk & 1][h], a0, a1, a2, a3, pf[0]);
              mma_bf16(c[2][h], a0, a1, a2, a3, pf[16 * KB * 32]);
              mma_bf16(c[3][h], a0, a1, a2, a3, pf[2 * 16 * KB * 32]);
            }
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < 4; ++r)
              zr[r >> 1][2 * h + (r & 1)] = (c[0][h][r] + c[1][h][r]) + (c[2][h][r] + c[3][h][r]);
        } else {
#pragma unroll
          for (int R = 0; R < 2; ++R) {
            const uint4 v = wb[(R * KB + a) * 32 + lane];
            zr[R][0] = __uint_as_float(v.x);
            zr[R][1] = __uint_as_float(v.y);
            zr[R][2] = __uint_as_float(v.z);
            zr[R][3] = __uint_as_float(v.w);
          }
        }
#pragma unroll
        for (int R = 0; R < 2; ++R) {
          float term[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // +0 for zero rows (never -0: the +0 addend)
            const float z = __fmaf_rn(zr[R][i], inv[R], 0.f);
            const int pos = 4 * hh + i;  // coordinate blk_base(a) + 8t + i is bit 8t + 4hh + i of word m
            if (corr) {
              // z and its centroid share a sign: z C = |z| |C|
              const uint2 rec = code_record(z, lut);
              Wm[R] += rec.y << pos;
              term[i] = fabsf(z) * fabsf(__uint_as_float(rec.x));
            } else {
              Wm[R] += code_spread(z, lut) << pos;
            }
          }
          if (corr) spart[R] += (term[0] + term[1]) + (term[2] + term[3]);
        }
      }
      if (corr) {
        ssum[0] += spart[0];
        ssum[1] += spart[1];
      }
#pragma unroll
      for (int R = 0; R < 2; ++R) {
        const uint32_t word = quad_transpose(Wm[R], t);  // plane t of word m
        if (okrow[R] && t < BITS) {
          if constexpr (MODE == kFlat) {
            codes[(size_t)nrow[R] * BITS * 4 + t * 4 + m] = word;
          } else if (is_key) {
            reinterpret_cast<uint32_t*>(dst[R] + P.off_kcodes)[(t * 16 + slot[R]) * 4 + m] = word;
          } else {
            vword[R][m] = word;  // written into the coordinate-major planes after the loop
          }
        }
      }
    }

    if (corr) {
      // key scale s = d / sum z C (balanced trees of positive terms: depth 3 within a
      // word pair, 4 words, 2 across the quad)
#pragma unroll
      for (int R = 0; R < 2; ++R) {
        float a = ssum[R];
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        const float sc = zero[R] ? 0.f : (float)D / a;
        if (okrow[R] && t == 0) {
          if constexpr (MODE == kFlat) rnorms[nrow[R]] = sc;
          else reinterpret_cast<float*>(dst[R] + P.off_krnorm)[slot[R]] = sc;
        }
      }
    }

    if constexpr (MODE == kStep) {
      if (!is_key) {
        // coordinate-major value planes: bit slot of the 16-bit entry (plane t, coordinate
        // j), one 32-bit word per coordinate pair.  Lane t rewrites its plane's 256 bytes
        // of the row's sub-block with two 16-byte accesses per word group; nothing else
        // writes them in this launch (one token per sequence, pages not shared).
#pragma unroll 1
        for (int R = 0; R < 2; ++R) {
          if (!okrow[R] || t >= BITS) continue;
          uint4* pl = reinterpret_cast<uint4*>(dst[R] + P.off_vcodes + (size_t)t * D * 2);
          uint4 wv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) wv[i] = pl[i];
          const int sl = slot[R];
          const uint32_t keep = ~((1u << sl) | (1u << (sl + 16)));
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t cw = vword[R][i >> 2];  // coordinates 32 (i / 4) .. + 31
            uint32_t e[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int c = 8 * (i & 3) + 2 * k;  // pair (c, c + 1) of the word
              e[k] = (e[k] & keep) | (((cw >> c) & 1u) << sl) | (((cw >> (c + 1)) & 1u) << (sl + 16));
            }
            pl[i] = make_uint4(e[0], e[1], e[2], e[3]);
          }
        }
      }
    }

    __syncwarp();  // the block buffer is rewritten by the next tile
  }
}


// ------------------------------------------------------------------ keys: QJL sketch on tcgen05
//
// Keys with the QJL sketch.  A CTA of 8 warps owns 128 vectors per pass (one
// UMMA M = 128 tile): every warp rotates, codes and packs its 16 vectors as in
// quantize_warp_kernel and writes the residual's f16 hi / lo limbs into the A
// tiles; one thread then issues S r as tcgen05.mma kind::f16 (hi*hi + hi*lo +
// lo*hi, fp32 accumulator of 128 x 128 in tensor memory) and the epilogue
// reads one vector per thread (tcgen05.ld 32x32b), packs its sign words and
// recomputes the uncertain entries in fp32 from the limbs in shared memory.

constexpr int kTcWarps = 8;
constexpr size_t kUmmaTile = (size_t)128 * 128 * 2;  // one 128 x 128 16-bit operand

// Canonical K-major operand without swizzle: 8 x 8 core matrices of 16-byte
// rows; K-chunk stride 128 B (leading byte offset), 8-row group stride 2048 B
// (stride byte offset).
__host__ __device__ constexpr uint32_t umma_off(int row, int k) {
  return (uint32_t)((row >> 3) * 2048 + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(2048 >> 4) << 32) |
         ((uint64_t)1 << 46);  // descriptor version 1, no swizzle
}

struct TcShared {
  float snorm[D];      // ||S_c|| (rounded up)
  float s2[128];       // ||r||^2 of each row (z units)
  uint32_t rec[128];   // flat: record index; step: page * Hkv + head
  uint8_t slot[128];   // step: slot in the page
  uint8_t flags[128];  // bit 0 row holds a vector, bit 1 zero vector
  uint64_t mbar;
  uint32_t tmem;
};

__host__ __device__ constexpr size_t tc_rest_bytes(bool dense) {
  return dense ? kPfragBytes : (size_t)KB * 2 * 32 * sizeof(uint2) + (size_t)kTcWarps * kBlkBytes;
}
__host__ __device__ constexpr size_t tc_smem_bytes(bool dense) {
  return 4 * kUmmaTile + tc_rest_bytes(dense) + sizeof(TcShared);  // + lut_bytes(J)
}

template <int BITS, bool DENSE, int MODE>
__global__ void __launch_bounds__(32 * kTcWarps, 1)
    quantize_keys_tc_kernel(const __grid_constant__ KParams P, const __grid_constant__ KCache C,
                            const __nv_bfloat16* __restrict__ x, long long n_vec, uint32_t* __restrict__ codes,
                            uint32_t* __restrict__ signs, float* __restrict__ norms, float* __restrict__ rnorms,
                            int lut_j, int tp) {
  constexpr int WARPS = kTcWarps;
  constexpr int NT = 32 * WARPS;
  extern __shared__ __align__(16) unsigned char smem_raw[];  // the no-swizzle operand layout needs 16-byte alignment
  unsigned char* Ahi = smem_raw;
  unsigned char* Alo = smem_raw + kUmmaTile;
  unsigned char* Bhi = smem_raw + 2 * kUmmaTile;
  unsigned char* Blo = smem_raw + 3 * kUmmaTile;
  unsigned char* rest = smem_raw + 4 * kUmmaTile;
  uint2* pfrag = reinterpret_cast<uint2*>(rest);                                     // dense: [3][16][KB][32]
  uint2* hfrag = reinterpret_cast<uint2*>(rest);                                     // FWHT: [KB][2][32]
  uint4* blk = reinterpret_cast<uint4*>(rest + (size_t)KB * 2 * 32 * sizeof(uint2));  // FWHT: [WARPS][2][KB][32]
  TcShared& ts = *reinterpret_cast<TcShared*>(rest + tc_rest_bytes(DENSE));
  unsigned char* lut_at = rest + tc_rest_bytes(DENSE) + sizeof(TcShared);  // code cell table and records

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int head = blockIdx.y;
  const float* rot = P.k_rot + (size_t)head * (DENSE ? D * D : D);
  // Gaussian S: [D][D] rows; structured S = H diag(sigma_S): the D signs, entries synthesised
  const float* S = P.qjl_s + (size_t)head * (P.qjl_srht ? D : D * D);
  build_code_lut<BITS, false>(lut_at, lut_j, P.kt, P.kc, tid, NT);
  const CodeLut lut = code_lut_at(lut_at, lut_j);

  if (warp == 0) {  // tensor memory: the 128 x 128 fp32 accumulator of S r
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ts.tmem)),
                 "r"(128));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&ts.mbar)), "r"(1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---- per-CTA constants: rotation fragments (mma.sync), S limbs (UMMA B tiles), ||S_c||
  if constexpr (!DENSE) {
    for (int i = tid; i < KB * 2 * 32; i += NT) {
      const int ln = i & 31, nt = (i >> 5) & 1, kk = i >> 6;
      const int gg = ln >> 2, tt = ln & 3;
      const float4 sg = __ldg(reinterpret_cast<const float4*>(rot + blk_base(kk) + 8 * tt));
      const float sv[4] = {sg.x, sg.y, sg.z, sg.w};
      const int out = 8 * (gg >> 1) + 2 * nt + (gg & 1);
      uint32_t h[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int L = 2 * tt + (e & 1) + 8 * (e >> 1);
        const bool neg = (sv[e] < 0.f) != (bool)(__popc(free_off(L) & out) & 1);
        h[e] = neg ? 0xBF80u : 0x3F80u;
      }
      hfrag[(kk * 2 + nt) * 32 + ln] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    }
  } else {
    constexpr int PER = (16 * KB * 32 + NT - 1) / NT;
    float4 pv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT;
      const int ln = i & 31, kk = (i >> 5) & (KB - 1), nt = (i >> 8) & 15;
      pv[j] = i < 16 * KB * 32
                  ? __ldg(reinterpret_cast<const float4*>(rot + (size_t)rot_out(nt, ln >> 2) * D + blk_base(kk) + 8 * (ln & 3)))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT;
      if (i >= 16 * KB * 32) break;
      const int ln = i & 31, kk = (i >> 5) & (KB - 1), nt = i >> 8;
      const float v[4] = {pv[j].x, pv[j].y, pv[j].z, pv[j].w};
      uint32_t l[3][4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float l0 = __bfloat162float(__float2bfloat16_rn(v[e]));
        const float l1 = __bfloat162float(__float2bfloat16_rn(v[e] - l0));
        l[0][e] = bf16_bits(v[e]);
        l[1][e] = bf16_bits(v[e] - l0);
        l[2][e] = bf16_bits((v[e] - l0) - l1);
      }
#pragma unroll
      for (int k = 0; k < 3; ++k)
        pfrag[((k * 16 + nt) * KB + kk) * 32 + ln] = make_uint2(l[k][0] | (l[k][1] << 16), l[k][2] | (l[k][3] << 16));
    }
  }
  {
    // S as UMMA B operands: row c of S (sketch coordinate), K = input coordinate
    constexpr int PER = 128 * 32 / NT;  // float4 chunks per thread
    float4 sv[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT, c = i >> 5, k0 = 4 * (i & 31);
      if (P.qjl_srht) {  // S[c][k] = (-1)^popcount(c & k) sigma_S[k], exact in f16 (lo limb 0)
        const float4 sg = __ldg(reinterpret_cast<const float4*>(S) + (i & 31));
        sv[j] = make_float4((__popc(c & k0) & 1) ? -sg.x : sg.x, (__popc(c & (k0 + 1)) & 1) ? -sg.y : sg.y,
                            (__popc(c & (k0 + 2)) & 1) ? -sg.z : sg.z, (__popc(c & (k0 + 3)) & 1) ? -sg.w : sg.w);
      } else {
        sv[j] = __ldg(reinterpret_cast<const float4*>(S + (size_t)c * D) + (i & 31));
      }
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT, c = i >> 5, k0 = 4 * (i & 31);
      const float v[4] = {sv[j].x, sv[j].y, sv[j].z, sv[j].w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = f16_bits(v[e]);
        lo[e] = f16_bits(v[e] - __half2float(__float2half_rn(v[e])));
      }
      *reinterpret_cast<uint2*>(Bhi + umma_off(c, k0)) = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
      *reinterpret_cast<uint2*>(Blo + umma_off(c, k0)) = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    }
    for (int c = tid; c < D; c += NT) {
      if (P.qjl_srht) {  // +-1 rows
        ts.snorm[c] = sqrtf((float)D) * 1.0001f;
        continue;
      }
      const float4* row = reinterpret_cast<const float4*>(S + (size_t)c * D);
      float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
      for (int i = 0; i < D / 4; ++i) {
        const float4 v = __ldg(row + i);
        acc4.x = fmaf(v.x, v.x, acc4.x);
        acc4.y = fmaf(v.y, v.y, acc4.y);
        acc4.z = fmaf(v.z, v.z, acc4.z);
        acc4.w = fmaf(v.w, v.w, acc4.w);
      }
      ts.snorm[c] = sqrtf((acc4.x + acc4.y) + (acc4.z + acc4.w)) * 1.0001f;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = ts.tmem;
  float smax = 0.f;
  for (int c = 0; c < D; ++c) smax = fmaxf(smax, ts.snorm[c]);

  // ---- passes over 128 vectors (8 warp tiles of 16 tokens of this head)
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 15) / 16;
  // a pass covers tp warp tiles (tp = WARPS for bulk calls; fewer spread a small decode-step
  // append over more CTAs): warp w < tp takes tile ct tp + w, the others hold no rows
  const long long n_ct = (n_tiles + tp - 1) / tp;
  auto warp_tile = [&](long long ct) -> long long { return warp < tp ? ct * tp + warp : n_tiles; };
  uint4* wb = blk + (size_t)warp * 2 * KB * 32;  // FWHT: this warp's rotated tile
  // |three-limb f16 product - exact product of the fp32 values|
  //   <= k1 ||r|| ||S_c|| + k2 (||r|| + ||S_c||):
  // k1 covers the dropped lo*lo term and the limb roundings (3 * 2^-22) and
  // the fp32 accumulation over 24 chained MMA steps even if every step
  // truncated each of its 17 addends by one unit in the last place
  // (24 * 17 * 2^-23); k2 covers f16 subnormal limbs (2^-25 per element,
  // times sqrt(d))
  const float k1 = 6e-5f, k2 = 4e-7f;
  // instruction descriptor: D f32, A and B f16, both K-major, N = 128, M = 128
  const uint32_t idesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

  auto row_index = [&](long long mt, int R, long long& n) -> bool {
    const long long tok = mt * 16 + g + 8 * R;
    n = tok * P.hkv + head;
    return tok < n_tok && n < n_vec;
  };
  uint4 nxt[2][4];
  auto load = [&](long long mt) {
#pragma unroll
    for (int R = 0; R < 2; ++R) {
      long long n;
      const bool ok = row_index(mt, R, n);
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(ok ? n : 0) * P.dh) + t;  // zero-padded to D
#pragma unroll
      for (int m = 0; m < 4; ++m) nxt[R][m] = (ok && 32 * m + 8 * t < P.dh) ? __ldg(src + 4 * m) : make_uint4(0, 0, 0, 0);
    }
  };
  uint32_t phase = 0;
  bool failed = false;
  if (blockIdx.x < n_ct) load(warp_tile(blockIdx.x));
  for (long long ct = blockIdx.x; ct < n_ct && !failed; ct += gridDim.x) {
    const long long mt = warp_tile(ct);
    uint4 X[2][4];
#pragma unroll
    for (int R = 0; R < 2; ++R)
#pragma unroll
      for (int m = 0; m < 4; ++m) X[R][m] = nxt[R][m];
    if (ct + gridDim.x < n_ct) load(warp_tile(ct + gridDim.x));

    long long nrow[2];
    bool okrow[2];
    unsigned char* dst[2] = {nullptr, nullptr};
    uint32_t recv[2] = {0u, 0u};
    int slot[2] = {0, 0};
#pragma unroll
    for (int R = 0; R < 2; ++R) {
      okrow[R] = row_index(mt, R, nrow[R]);
      recv[R] = (uint32_t)nrow[R];
      if constexpr (MODE == kStep) {
        if (okrow[R]) {
          const int b = (int)(nrow[R] / P.hkv);
          const int T = C.seq_len[b];
          const int pidx = T >> 4;
          long long page = -1;
          if (T >= 0 && pidx < C.max_pages) page = C.block_table[(size_t)b * C.max_pages + pidx];
          if (page < 0 || page >= C.n_pages) {
            if (t == 0) atomicOr(&g_quant_err, (T >= 0 && pidx < C.max_pages) ? TQ_DEVERR_PAGE_INDEX : TQ_DEVERR_SEQ_LEN);
            okrow[R] = false;
          } else {
            recv[R] = (uint32_t)(page * P.hkv + head);
            dst[R] = C.pool + (size_t)recv[R] * (size_t)P.sub_bytes;
            slot[R] = T & 15;
          }
        }
      }
    }

    // norms (balanced fp32 tree over exact bf16 squares)
    float inv[2];
    bool zero[2];
#pragma unroll
    for (int R = 0; R < 2; ++R) {
      float part[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t w[4] = {X[R][m].x, X[R][m].y, X[R][m].z, X[R][m].w};
        float q2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
          q2[k] = lo * lo + hi * hi;
        }
        part[m] = (q2[0] + q2[1]) + (q2[2] + q2[3]);
      }
      float s2 = (part[0] + part[1]) + (part[2] + part[3]);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
      const float n = sqrtf(s2);
      zero[R] = n < kZeroNorm;
      inv[R] = zero[R] ? 0.f : sqrtf((DENSE ? (float)D : 1.0f) / s2);
      if (okrow[R] && t == 0) {
        if constexpr (MODE == kFlat) norms[nrow[R]] = zero[R] ? 0.f : n;
        else reinterpret_cast<float*>(dst[R] + P.off_knorm)[slot[R]] = zero[R] ? 0.f : n;
      }
    }

    if constexpr (!DENSE) {
      float acc[KB][2][4];
#pragma unroll
      for (int kk = 0; kk < KB; ++kk) {
        const uint4& u0 = X[0][kk >> 1];
        const uint4& u1 = X[1][kk >> 1];
        const uint32_t a0 = (kk & 1) ? u0.z : u0.x, a2 = (kk & 1) ? u0.w : u0.y;
        const uint32_t a1 = (kk & 1) ? u1.z : u1.x, a3 = (kk & 1) ? u1.w : u1.y;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[kk][h][r] = 0.f;
          mma_bf16(acc[kk][h], a0, a1, a2, a3, hfrag[(kk * 2 + h) * 32 + lane]);
        }
      }
#pragma unroll
      for (int s = 1; s < KB; s <<= 1)
#pragma unroll
        for (int a = 0; a < KB; ++a)
          if ((a & s) == 0)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const float p = acc[a][h][r], q = acc[a + s][h][r];
                acc[a][h][r] = p + q;
                acc[a + s][h][r] = p - q;
              }
#pragma unroll
      for (int a = 0; a < KB; ++a) {
        wb[(0 * KB + a) * 32 + lane] = make_uint4(__float_as_uint(acc[a][0][0]), __float_as_uint(acc[a][0][1]),
                                                  __float_as_uint(acc[a][1][0]), __float_as_uint(acc[a][1][1]));
        wb[(1 * KB + a) * 32 + lane] = make_uint4(__float_as_uint(acc[a][0][2]), __float_as_uint(acc[a][0][3]),
                                                  __float_as_uint(acc[a][1][2]), __float_as_uint(acc[a][1][3]));
      }
    }

    // codes and the residual limbs (A tiles), two blocks per pass
    float rs[2] = {0.f, 0.f};
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      uint32_t Wm[2] = {0u, 0u};
      float pr[2] = {0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int a = 2 * m + hh;
        float zr[2][4];
        if constexpr (DENSE) {
          float c[4][2][4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int r = 0; r < 4; ++r) c[i][h][r] = 0.f;
#pragma unroll
          for (int kk = 0; kk < KB; ++kk) {
            const uint4& u0 = X[0][kk >> 1];
            const uint4& u1 = X[1][kk >> 1];
            const uint32_t a0 = (kk & 1) ? u0.z : u0.x, a2 = (kk & 1) ? u0.w : u0.y;
            const uint32_t a1 = (kk & 1) ? u1.z : u1.x, a3 = (kk & 1) ? u1.w : u1.y;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint2* pf = pfrag + ((2 * a + h) * KB + kk) * 32 + lane;
              mma_bf16(c[kk & 1][h], a0, a1, a2, a3, pf[0]);
              mma_bf16(c[2][h], a0, a1, a2, a3, pf[16 * KB * 32]);
              mma_bf16(c[3][h], a0, a1, a2, a3, pf[2 * 16 * KB * 32]);
            }
          }
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int r = 0; r < 4; ++r)
              zr[r >> 1][2 * h + (r & 1)] = (c[0][h][r] + c[1][h][r]) + (c[2][h][r] + c[3][h][r]);
        } else {
#pragma unroll
          for (int R = 0; R < 2; ++R) {
            const uint4 v = wb[(R * KB + a) * 32 + lane];
            zr[R][0] = __uint_as_float(v.x);
            zr[R][1] = __uint_as_float(v.y);
            zr[R][2] = __uint_as_float(v.z);
            zr[R][3] = __uint_as_float(v.w);
          }
        }
        float rv[2][4];
#pragma unroll
        for (int R = 0; R < 2; ++R)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float z = __fmaf_rn(zr[R][i], inv[R], 0.f);
            const uint2 rec = code_record(z, lut);
            Wm[R] += rec.y << (4 * hh + i);
            rv[R][i] = z - __uint_as_float(rec.x);
          }
        const int j0 = blk_base(a) + 8 * t;  // this lane's four coordinates of block a
#pragma unroll
        for (int R = 0; R < 2; ++R) {
          const int row = 16 * warp + g + 8 * R;
          const uint32_t h01 = pack_f16(rv[R][0], rv[R][1]), h23 = pack_f16(rv[R][2], rv[R][3]);
          *reinterpret_cast<uint2*>(Ahi + umma_off(row, j0)) = make_uint2(h01, h23);
          *reinterpret_cast<uint2*>(Alo + umma_off(row, j0)) =
              make_uint2(pack_f16(rv[R][0] - f16lo(h01), rv[R][1] - f16hi(h01)),
                         pack_f16(rv[R][2] - f16lo(h23), rv[R][3] - f16hi(h23)));
          pr[R] += (rv[R][0] * rv[R][0] + rv[R][1] * rv[R][1]) + (rv[R][2] * rv[R][2] + rv[R][3] * rv[R][3]);
        }
      }
#pragma unroll
      for (int R = 0; R < 2; ++R) {
        rs[R] += pr[R];
        const uint32_t word = quad_transpose(Wm[R], t);
        if (okrow[R] && t < BITS) {
          if constexpr (MODE == kFlat) codes[(size_t)nrow[R] * BITS * 4 + t * 4 + m] = word;
          else reinterpret_cast<uint32_t*>(dst[R] + P.off_kcodes)[(t * 16 + slot[R]) * 4 + m] = word;
        }
      }
    }
#pragma unroll
    for (int R = 0; R < 2; ++R) {
      float s2 = rs[R];
      s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
      if (t == 0) {
        const int row = 16 * warp + g + 8 * R;
        ts.s2[row] = s2;
        ts.rec[row] = recv[R];
        ts.slot[row] = (uint8_t)slot[R];
        ts.flags[row] = (uint8_t)((okrow[R] ? 1 : 0) | (zero[R] ? 2 : 0));
      }
    }

    // ---- S r on the tensor cores: 3 limb products x 8 k-steps into tensor memory
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (tid == 0) {
      const uint32_t a_hi = smem_u32(Ahi), a_lo = smem_u32(Alo), b_hi = smem_u32(Bhi), b_lo = smem_u32(Blo);
      const uint32_t as_[3] = {a_hi, a_hi, a_lo}, bs_[3] = {b_hi, b_lo, b_hi};
#pragma unroll
      for (int pss = 0; pss < 3; ++pss)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t accum = (pss > 0 || ks > 0) ? 1u : 0u;
          asm volatile(
              "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
              " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
              "l"(umma_desc(as_[pss] + 256 * ks)), "l"(umma_desc(bs_[pss] + 256 * ks)), "r"(idesc), "r"(accum));
        }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(&ts.mbar)));
    }
    uint32_t done = 0;
    for (unsigned it = 0; it < (1u << 22) && !done; ++it) {
      asm volatile(
          "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
          : "=r"(done)
          : "r"(smem_u32(&ts.mbar)), "r"(phase));
    }
    phase ^= 1u;
    if (__syncthreads_or(!done)) {  // the sketch never completed: flag it, stop cleanly
      if (tid == 0) atomicOr(&g_quant_err, TQ_DEVERR_TIMEOUT);
      failed = true;
      break;
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // ---- epilogue: vector row = 32 (warp % 4) + lane, sketch coordinates 64 (warp / 4) .. + 63
    {
      const int row = 32 * (warp & 3) + lane, hcol = 64 * (warp >> 2);
      const uint32_t fl = ts.flags[row];
      const bool ok = fl & 1u, zr = fl & 2u;
      const float s2 = ts.s2[row];
      const float rn = sqrtf(s2);
      const float bA = fmaf(k1, rn, k2), bB = fmaf(k2, rn, k2);
      const float bmax = fmaf(smax, bA, bB);  // the bound of the row's largest ||S_c||, for every c
      const uint32_t rec = ts.rec[row];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c0 = hcol + 32 * cc;
        uint32_t v[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
            "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
              "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)c0));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        // raw sign bits and "uncertain" bits, highest coordinate first through a
        // funnel shift; -0 reads as negative but is always uncertain (bound > 0)
        uint32_t neg = 0, pend = 0;
#pragma unroll
        for (int j = 31; j >= 0; --j) {
          uint32_t lt;
          asm("set.lt.u32.f32 %0, %1, %2;" : "=r"(lt) : "f"(fabsf(__uint_as_float(v[j]))), "f"(bmax));
          asm("shf.l.wrap.b32 %0, %1, %2, 1;" : "=r"(neg) : "r"(v[j]), "r"(neg));
          asm("shf.l.wrap.b32 %0, %1, %2, 1;" : "=r"(pend) : "r"(lt), "r"(pend));
        }
        uint32_t word = ~neg;
        if (zr) {
          word = 0xffffffffu;
          pend = 0u;
        }
        if (!ok) pend = 0u;
        // fp32 recomputation of the uncertain entries from the limbs, one entry per
        // pass of the warp (a few per thousand vectors); lane l covers coordinates 4l .. 4l + 3
        while (true) {
          const unsigned ball = __ballot_sync(0xffffffffu, pend != 0u);
          if (ball == 0u) break;
          const int src = __ffs(ball) - 1;
          const int j = __shfl_sync(0xffffffffu, __ffs(pend) - 1, src);
          const int frow = 32 * (warp & 3) + src, c = c0 + j, k0 = 4 * lane;
          const uint2 ah = *reinterpret_cast<const uint2*>(Ahi + umma_off(frow, k0));
          const uint2 al = *reinterpret_cast<const uint2*>(Alo + umma_off(frow, k0));
          const uint2 bh = *reinterpret_cast<const uint2*>(Bhi + umma_off(c, k0));
          const uint2 bl = *reinterpret_cast<const uint2*>(Blo + umma_off(c, k0));
          float dsum = (f16lo(ah.x) + f16lo(al.x)) * (f16lo(bh.x) + f16lo(bl.x));
          dsum = fmaf(f16hi(ah.x) + f16hi(al.x), f16hi(bh.x) + f16hi(bl.x), dsum);
          dsum = fmaf(f16lo(ah.y) + f16lo(al.y), f16lo(bh.y) + f16lo(bl.y), dsum);
          dsum = fmaf(f16hi(ah.y) + f16hi(al.y), f16hi(bh.y) + f16hi(bl.y), dsum);
          dsum = warp_sum_f(dsum);
          if (lane == src) {
            word = (word & ~(1u << j)) | ((uint32_t)(dsum >= 0.f) << j);
            pend &= ~(1u << j);
          }
        }
        if (ok) {
          const int wi = 2 * (warp >> 2) + cc;  // sign word index
          if constexpr (MODE == kFlat) signs[(size_t)rec * 4 + wi] = word;
          else reinterpret_cast<uint32_t*>(C.pool + (size_t)rec * P.sub_bytes + P.off_ksigns)[ts.slot[row] * 4 + wi] = word;
        }
      }
      if (ok && (warp >> 2) == 0) {
        const float gam = zr ? 0.f : sqrtf(s2 * (1.0f / D));  // exact scaling by a power of two
        if constexpr (MODE == kFlat) rnorms[rec] = gam;
        else reinterpret_cast<float*>(C.pool + (size_t)rec * P.sub_bytes + P.off_krnorm)[ts.slot[row]] = gam;
      }
    }
    // the A tiles, the row table and the accumulator are rewritten by the next pass
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
  }
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(128));
}

}  // namespace wq
}  // namespace tq
