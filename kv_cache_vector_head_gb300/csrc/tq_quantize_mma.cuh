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
//   * QJL: S r as three f16 MMAs over hi / lo limbs of r and S (hi*hi +
//     hi*lo + lo*hi).  Every entry whose magnitude is below a certified
//     bound of the limb and accumulation errors (6e-5 ||r|| ||S_c||, a few
//     per thousand vectors) is recomputed in fp32 by the warp from the
//     limbs, so every sign is that of the fp32 product up to 2^-21 relative;
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

#include "tq_device.cuh"

namespace tq {

// The including file defines tq::g_quant_err (the device error word of the
// quantize / append kernels) before including this header.

namespace wq {

constexpr int D = 128;
constexpr int KB = D / 16;     // k-blocks

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
  float snorm[D];              // ||S_c|| (rounded up)
  uint2 hfrag[KB][2][32];      // FWHT H_16 * sigma fragments (bf16)
};
constexpr size_t kSfragBytes = (size_t)2 * 16 * KB * 32 * sizeof(uint2);  // S as f16 hi and lo limbs
constexpr size_t kPfragBytes = (size_t)3 * 16 * KB * 32 * sizeof(uint2);  // Pi limbs (bf16)
// Per-warp block buffer: [2][KB][32] uint4.  FWHT: the rotated tile (R = 0
// rows in half 0, R = 1 rows in half 1); keys: then the residual's f16 hi
// and lo limbs in A-fragment order, written over the same slots.
constexpr size_t kBlkBytes = (size_t)2 * KB * 32 * sizeof(uint4);

// FWHT: 12 warps, next tile staged in shared memory by cp.async; dense: the
// Pi limbs fill most of shared memory (7 warps with the sketch, 8 and two
// CTAs per SM without), next tile prefetched into registers.
__host__ __device__ constexpr int warps_for(bool qjl, bool dense) { return dense ? (qjl ? 7 : 8) : 12; }
__host__ __device__ constexpr int ctas_for(bool qjl, bool dense) { return dense && !qjl ? 2 : 1; }
__host__ __device__ constexpr size_t blk_bytes(bool qjl, bool dense) {
  return (qjl || !dense) ? (size_t)warps_for(qjl, dense) * kBlkBytes : 0;
}
__host__ __device__ constexpr size_t stage_bytes(bool qjl, bool dense) {
  return dense ? 0 : (size_t)warps_for(qjl, dense) * 8 * 32 * sizeof(uint4);
}

__host__ __device__ constexpr size_t smem_bytes(bool qjl, bool dense) {
  return sizeof(Shared) + (qjl ? kSfragBytes : 0) + (dense ? kPfragBytes : 0) + blk_bytes(qjl, dense) +
         stage_bytes(qjl, dense);
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

// Positive half of an antisymmetric codebook: boundaries (as int bits,
// ascending) and centroids.
template <int BITS>
struct Book {
  int tp[BITS > 1 ? (1 << (BITS - 1)) - 1 : 1];
  float cp[1 << (BITS - 1)];
};

// Number of positive boundaries t with ai >= bits(t) (binary search).
template <int BITS>
__device__ __forceinline__ int magnitude(int ai, const Book<BITS>& b) {
  if constexpr (BITS == 1) {
    return 0;
  } else if constexpr (BITS == 2) {
    return ai >= b.tp[0] ? 1 : 0;
  } else if constexpr (BITS == 3) {
    const int m1 = ai >= b.tp[1] ? 2 : 0;
    return m1 + (ai >= (m1 ? b.tp[2] : b.tp[0]) ? 1 : 0);
  } else {
    const int m2 = ai >= b.tp[3] ? 4 : 0;
    const int m1 = ai >= (m2 ? b.tp[5] : b.tp[1]) ? 2 : 0;
    const int th = m2 ? (m1 ? b.tp[6] : b.tp[4]) : (m1 ? b.tp[2] : b.tp[0]);
    return m2 + m1 + (ai >= th ? 1 : 0);
  }
}

template <int BITS>
__device__ __forceinline__ float centroid_pos(int mag, const Book<BITS>& b) {
  float c = b.cp[0];
#pragma unroll
  for (int i = 1; i < (1 << (BITS - 1)); ++i) c = mag == i ? b.cp[i] : c;
  return c;
}

__device__ __forceinline__ float f16lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// Where the records go: flat arrays (bulk quantize) or the page slot of each
// sequence's next token (decode-step append without a window: rows are the
// sequences, the token of sequence b lands in slot seq_len[b] % 16 of page
// block_table[b][seq_len[b] / 16]).
enum { kFlat = 0, kStep = 1 };

// QJL: keys with the sketch; DENSE: dense rotation (else FWHT).  grid (x, Hkv).
template <int BITS, bool QJL, bool DENSE, int MODE>
__global__ void __launch_bounds__(32 * warps_for(QJL, DENSE), ctas_for(QJL, DENSE))
    quantize_warp_kernel(const __grid_constant__ KParams P, const __grid_constant__ KCache C,
                         const __nv_bfloat16* __restrict__ x, long long n_vec, int is_key,
                         uint32_t* __restrict__ codes, uint32_t* __restrict__ signs, float* __restrict__ norms,
                         float* __restrict__ rnorms) {
  constexpr int WARPS = warps_for(QJL, DENSE);
  constexpr int NT = 32 * WARPS;
  constexpr int HALF = 1 << (BITS - 1);
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  unsigned char* dyn = smem_raw + sizeof(Shared);
  uint2* sfrag = reinterpret_cast<uint2*>(dyn);  // [2 limbs][16][KB][32]
  dyn += QJL ? kSfragBytes : 0;
  uint2* pfrag = reinterpret_cast<uint2*>(dyn);  // [3][16][KB][32]
  dyn += DENSE ? kPfragBytes : 0;
  uint4* blk = reinterpret_cast<uint4*>(dyn);    // [WARPS][2][KB][32]
  dyn += blk_bytes(QJL, DENSE);
  uint4* stage = reinterpret_cast<uint4*>(dyn);  // [WARPS][8][32]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, t = lane & 3;
  const int head = blockIdx.y;
  const float* ctab = is_key ? P.kc : P.vc;
  const float* ttab = is_key ? P.kt : P.vt;
  const float* rot = (is_key ? P.k_rot : P.v_rot) + (size_t)head * (DENSE ? D * D : D);
  const float* S = QJL ? P.qjl_s + (size_t)head * D * D : nullptr;
  Book<BITS> bk;
#pragma unroll
  for (int k = 0; k + 1 < HALF; ++k) bk.tp[k] = __float_as_int(ttab[HALF + k]);
#pragma unroll
  for (int m = 0; m < HALF; ++m) bk.cp[m] = ctab[HALF + m];

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
  if constexpr (QJL) {
    constexpr int PER = (16 * KB * 32 + NT - 1) / NT;
    float4 sv4[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT;
      const int ln = i & 31, kk = (i >> 5) & (KB - 1), nt = (i >> 8) & 15;
      sv4[j] = i < 16 * KB * 32
                   ? __ldg(reinterpret_cast<const float4*>(S + (size_t)sk_out(nt, ln >> 2) * D + blk_base(kk) + 8 * (ln & 3)))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = tid + j * NT;
      if (i >= 16 * KB * 32) break;
      const int ln = i & 31, kk = (i >> 5) & (KB - 1), nt = i >> 8;
      const float4 v4 = sv4[j];
      const float v[4] = {v4.x, v4.y, v4.z, v4.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = f16_bits(v[e]);
        lo[e] = f16_bits(v[e] - __half2float(__float2half_rn(v[e])));
      }
      sfrag[(nt * KB + kk) * 32 + ln] = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
      sfrag[((16 + nt) * KB + kk) * 32 + ln] = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    }
    // ||S_c||: thread c sums its row from the fragments' source (fp32, L2-hot)
    for (int c = tid; c < D; c += NT) {
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
      sh.snorm[c] = sqrtf((acc4.x + acc4.y) + (acc4.z + acc4.w)) * 1.0001f;
    }
  }
  __syncthreads();

  // ---- tiles of 16 tokens of this head
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 15) / 16;
  const long long stride = (long long)gridDim.x * WARPS;
  uint4* wb = blk + (size_t)warp * 2 * KB * 32;  // this warp's block buffer: wb[(half * KB + a) * 32 + lane]
  // |three-limb f16 product - exact product of the fp32 values|
  //   <= k1 ||r|| ||S_c|| + k2 (||r|| + ||S_c||):
  // k1 covers the dropped lo*lo term and the limb roundings (3 * 2^-22) and
  // the fp32 accumulation over 24 chained MMAs even if every MMA truncated
  // each of its 17 addends by one unit in the last place (24 * 17 * 2^-23);
  // k2 covers f16 subnormal limbs (2^-25 per element, times sqrt(d))
  const float k1 = 6e-5f, k2 = 4e-7f;

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
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)(ok ? n : 0) * D) + t;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        if constexpr (DENSE) nxt[R][m] = ok ? __ldg(src + 4 * m) : make_uint4(0, 0, 0, 0);
        else cp_async16(stg + 32 * (4 * R + m), src + 4 * m, ok ? 16 : 0);
      }
    }
    if constexpr (!DENSE) cp_async_commit();
  };
  long long mt = (long long)blockIdx.x * WARPS + warp;
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
    float rs[2] = {0.f, 0.f};  // ||r||^2: block sums, pairs, then the four words in turn
    uint32_t vword[2][4];      // step mode, values: plane t of words 0..3 of rows g, g + 8
#pragma unroll 1
    for (int m = 0; m < 4; ++m) {
      uint32_t Wm[2] = {0u, 0u};  // byte p: plane p of this lane's byte of word m
      float pr[2] = {0.f, 0.f};
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
        float rv[2][4];
#pragma unroll
        for (int R = 0; R < 2; ++R)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float z = __fmaf_rn(zr[R][i], inv[R], 0.f);  // +0 for zero rows
            const uint32_t zb = __float_as_uint(z);
            const uint32_t neg = zb >> 31;
            const int ai = (int)(zb & 0x7fffffffu) - (int)neg;  // for z < 0: |z| > t <=> ai >= bits(t)
            const int mag = magnitude<BITS>(ai, bk);
            const uint32_t q = (neg ^ 1u) | ((uint32_t)mag << 1);
            const int pos = 4 * hh + i;  // coordinate blk_base(a) + 8t + i is bit 8t + 4hh + i of word m
            Wm[R] |= (q * (0x204081u << pos)) & (0x01010101u << pos);
            if constexpr (QJL) rv[R][i] = z - __uint_as_float(__float_as_uint(centroid_pos<BITS>(mag, bk)) ^ (neg << 31));
          }
        if constexpr (QJL) {
          // residual limbs in A-fragment order (rows g, g+8; coordinate pairs 8t+{0,1}, 8t+{2,3})
          const float2 p0 = make_float2(rv[0][0], rv[0][1]), p1 = make_float2(rv[1][0], rv[1][1]);
          const float2 p2 = make_float2(rv[0][2], rv[0][3]), p3 = make_float2(rv[1][2], rv[1][3]);
          const uint32_t h0 = pack_f16(p0.x, p0.y), h1 = pack_f16(p1.x, p1.y);
          const uint32_t h2 = pack_f16(p2.x, p2.y), h3 = pack_f16(p3.x, p3.y);
          wb[(0 * KB + a) * 32 + lane] = make_uint4(h0, h1, h2, h3);
          wb[(1 * KB + a) * 32 + lane] =
              make_uint4(pack_f16(p0.x - f16lo(h0), p0.y - f16hi(h0)), pack_f16(p1.x - f16lo(h1), p1.y - f16hi(h1)),
                         pack_f16(p2.x - f16lo(h2), p2.y - f16hi(h2)), pack_f16(p3.x - f16lo(h3), p3.y - f16hi(h3)));
#pragma unroll
          for (int R = 0; R < 2; ++R)
            pr[R] += (rv[R][0] * rv[R][0] + rv[R][1] * rv[R][1]) + (rv[R][2] * rv[R][2] + rv[R][3] * rv[R][3]);
        }
      }
#pragma unroll
      for (int R = 0; R < 2; ++R) {
        rs[R] += pr[R];
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

    if constexpr (QJL) {
      float gam[2], bA[2], bB[2];
#pragma unroll
      for (int R = 0; R < 2; ++R) {
        float s2 = rs[R];
        s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
        s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
        gam[R] = sqrtf(s2 * (1.0f / D));  // exact scaling by a power of two
        const float rn = sqrtf(s2);
        bA[R] = fmaf(k1, rn, k2);
        bB[R] = k2 * rn + k2;
      }
      uint32_t rA[KB][4];
#pragma unroll
      for (int a = 0; a < KB; ++a) {
        const uint4 v = wb[(0 * KB + a) * 32 + lane];
        rA[a][0] = v.x;
        rA[a][1] = v.y;
        rA[a][2] = v.z;
        rA[a][3] = v.w;
      }
      __syncwarp();  // residual limbs visible to the whole warp for the fp32 recomputations
      const uint32_t zmask = (zero[0] ? 0xffu : 0u) | (zero[1] ? 0xff00u : 0u);
      uint32_t SB[2] = {0u, 0u};
#pragma unroll 1
      for (int w = 0; w < 4; ++w) {
        float sacc[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int r = 0; r < 4; ++r) sacc[q][r] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KB; ++kk) {
          const uint4 lo = wb[(1 * KB + kk) * 32 + lane];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint2 bh = sfrag[((4 * w + q) * KB + kk) * 32 + lane];
            const uint2 bl = sfrag[((16 + 4 * w + q) * KB + kk) * 32 + lane];
            mma_f16(sacc[q], rA[kk][0], rA[kk][1], rA[kk][2], rA[kk][3], bh);
            mma_f16(sacc[q], rA[kk][0], rA[kk][1], rA[kk][2], rA[kk][3], bl);
            mma_f16(sacc[q], lo.x, lo.y, lo.z, lo.w, bh);
          }
        }
        const float4 sn0 = *reinterpret_cast<const float4*>(&sh.snorm[32 * w + 8 * t]);
        const float4 sn1 = *reinterpret_cast<const float4*>(&sh.snorm[32 * w + 8 * t + 4]);
        const float sn[8] = {sn0.x, sn0.y, sn0.z, sn0.w, sn1.x, sn1.y, sn1.z, sn1.w};
        uint32_t sb = 0, pend = 0;  // bit 8R + 2q + e
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int R = r >> 1, e = r & 1, bit = 8 * R + 2 * q + e;
            const float v = sacc[q][r];
            sb |= (uint32_t)(v >= 0.f) << bit;
            pend |= (uint32_t)(fabsf(v) < fmaf(sn[2 * q + e], bA[R], bB[R])) << bit;
          }
        sb |= zmask;
        pend &= ~zmask;
        // fp32 recomputation of the uncertain entries, one per pass of the warp,
        // from the f16 hi + lo limbs of r and S (22 bits each); lane l covers
        // coordinates blk_base(l / 4) + 8 (l % 4) + 0..3, which are one B
        // fragment of the sketch row
        while (true) {
          const unsigned ball = __ballot_sync(0xffffffffu, pend != 0);
          if (ball == 0) break;
          const int src = __ffs(ball) - 1;
          const int bit = __shfl_sync(0xffffffffu, __ffs(pend) - 1, src);
          const int row = (src >> 2) + 8 * (bit >> 3), R = row >> 3;
          const int nt = 4 * w + ((bit >> 1) & 3), n = 2 * (src & 3) + (bit & 1);  // sketch coordinate sk_out(nt, n)
          const int ab = lane >> 2, tl = lane & 3;
          const uint32_t* hi = reinterpret_cast<const uint32_t*>(wb + (0 * KB + ab) * 32 + (row & 7) * 4 + tl);
          const uint32_t* lo = reinterpret_cast<const uint32_t*>(wb + (1 * KB + ab) * 32 + (row & 7) * 4 + tl);
          const uint32_t h01 = hi[R], h23 = hi[2 + R], l01 = lo[R], l23 = lo[2 + R];
          const uint2 sh2 = sfrag[(nt * KB + ab) * 32 + 4 * n + tl];
          const uint2 sl2 = sfrag[((16 + nt) * KB + ab) * 32 + 4 * n + tl];
          float dsum = (f16lo(h01) + f16lo(l01)) * (f16lo(sh2.x) + f16lo(sl2.x));
          dsum = fmaf(f16hi(h01) + f16hi(l01), f16hi(sh2.x) + f16hi(sl2.x), dsum);
          dsum = fmaf(f16lo(h23) + f16lo(l23), f16lo(sh2.y) + f16lo(sl2.y), dsum);
          dsum = fmaf(f16hi(h23) + f16hi(l23), f16hi(sh2.y) + f16hi(sl2.y), dsum);
          dsum = warp_sum_f(dsum);
          if (lane == src) {
            sb = (sb & ~(1u << bit)) | ((uint32_t)(dsum >= 0.f) << bit);
            pend &= ~(1u << bit);
          }
        }
        SB[0] |= (sb & 0xffu) << (8 * w);
        SB[1] |= ((sb >> 8) & 0xffu) << (8 * w);
      }
#pragma unroll
      for (int R = 0; R < 2; ++R) {
        const uint32_t word = quad_transpose(SB[R], t);
        if constexpr (MODE == kFlat) {
          if (okrow[R]) signs[(size_t)nrow[R] * 4 + t] = word;
          if (okrow[R] && t == 0) rnorms[nrow[R]] = zero[R] ? 0.f : gam[R];
        } else {
          if (okrow[R]) reinterpret_cast<uint32_t*>(dst[R] + P.off_ksigns)[slot[R] * 4 + t] = word;
          if (okrow[R] && t == 0) reinterpret_cast<float*>(dst[R] + P.off_krnorm)[slot[R]] = zero[R] ? 0.f : gam[R];
        }
      }
    }
    __syncwarp();  // the block buffer is rewritten by the next tile
  }
}

}  // namespace wq
}  // namespace tq
