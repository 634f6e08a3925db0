// TurboQuant key / value quantization and paged append (sm_103a).
//
// [Reconstruction] §5 Steps 1-5 (norm separation, rotation, Lloyd-Max code)
// and §6 (residual, QJL sign sketch); [Design study] §CPU and WASM kernel
// design ("Append-time key kernel": sign flips + FWHT, quantize, pack, store
// norm and the residual sign stream), §Packed format, §Append cost.
//
// One CTA owns a tile of up to 16 vectors of ONE kv head (so the per-head
// rotation and QJL matrix are shared by the tile) and blockDim == d threads:
//   1. norms in double, one warp per vector;
//   2. rotation: FWHT as a register/shuffle butterfly, one warp per vector
//      (coordinate e*32 + lane lives in register e of that lane), or the dense
//      rotation as a tile product, thread j computing coordinate j of every
//      vector of the tile;
//   3. bucketize z = sqrt(d) * (Pi x) / n against the float32 boundaries and
//      pack sign-magnitude planes with warp ballots (warp w owns word w);
//   4. keys: residual (in z units) z - C[idx], its norm, and the QJL sketch
//      S (z - C[idx]) as a second tile product; signs packed by ballot.  The
//      scaled corrections keep s instead: EDEN's unbiased scale and TurboVec's
//      length-renormalized correction ([Reconstruction] §12 item 2, §13 step 6:
//      norm / <y, y_hat>, with the norm kept in its own field) are the same
//      number, s = 1 / <y, y_hat> = d / sum z C[idx].
// Mixed-channel keys ([Design study] §Packed format: fractional rates by
// channel allocation) take coordinates < d/2 one bit wider with their own
// book; the wider codes' top plane is kept for the first d/64 words only.
// Byte key norms (u8 log-norm) are encoded when the page slot is written.
// The structured sketch S = H diag(sigma_S) takes the signs of a warp
// Walsh-Hadamard transform of sigma_S * r instead of the tile product.
#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_launch.h"
#include "tq_tile.cuh"

namespace tq {
__device__ unsigned int g_quant_err = 0;
}  // namespace tq

#include "tq_quantize_mma.cuh"
#include "tq_quantize_tc.cuh"

namespace tq {

// Quantize the tile held in s.x (nv vectors, rows >= nv are ignored).
// is_key selects the key codebook/transform and the QJL stage.
// slot_of[v] (when non-null) gives the page slot of vector v for the
// coordinate-major value masks.  ONE: nv is 1 (a decode-step append), which takes its own sketch loop.
template <int D, bool ONE = false>
__device__ void quantize_tile(const KParams& P, TileSmem<D>& s, int nv, int head, bool is_key,
                              const int* slot_of) {
  constexpr int E = D / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int bits = is_key ? P.kb : P.vb;
  const bool split = is_key && P.ksplit;  // coordinates < d/2 one bit wider, own book
  const float sqrt_d = sqrtf((float)D);
  if (tid < 16) {
    s.cb[tid] = is_key ? P.kc[tid] : P.vc[tid];
    s.tb[tid] = is_key ? P.kt[tid] : P.vt[tid];
    s.cb_hi[tid] = P.kc_hi[tid];
    s.tb_hi[tid] = P.kt_hi[tid];
  }
  // 1. norms (double accumulation; one vector: float, pairwise, relative error below 13 ulp on the sum)
  if constexpr (ONE) {
    if (warp == 0) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc = fmaf(s.x[0][e * 32 + lane], s.x[0][e * 32 + lane], acc);
      acc = warp_sum_f(acc);  // the same in every lane
      if (acc >= 1e-30f && acc <= 1e37f) {
        if (lane == 0) {
          const float n = sqrtf(acc);
          const bool zero = n < kZeroNorm;
          s.zero[0] = zero;
          s.norm[0] = zero ? 0.f : n;
          s.inv[0] = zero ? 0.f : (P.kind == TQ_FWHT ? 1.f / n : sqrt_d / n);
        }
      } else {  // squares near the float range's ends (or a non-finite input): the double sum
        double dacc = 0.0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const double xv = s.x[0][e * 32 + lane];
          dacc += xv * xv;
        }
        dacc = warp_sum_d(dacc);
        if (lane == 0) {
          const double n = sqrt(dacc);
          const bool zero = n < (double)kZeroNorm;
          s.zero[0] = zero;
          s.norm[0] = zero ? 0.f : (float)n;
          s.inv[0] = zero ? 0.f : (P.kind == TQ_FWHT ? (float)(1.0 / n) : (float)((double)sqrt_d / n));
        }
      }
    }
  } else for (int v = warp; v < nv; v += D / 32) {
    double acc = 0.0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const double xv = s.x[v][e * 32 + lane];
      acc += xv * xv;
    }
    acc = warp_sum_d(acc);
    if (lane == 0) {
      const double n = sqrt(acc);
      const bool zero = n < (double)kZeroNorm;
      s.zero[v] = zero;
      s.norm[v] = zero ? 0.f : (float)n;
      s.inv[v] = zero ? 0.f : (P.kind == TQ_FWHT ? (float)(1.0 / n) : (float)((double)sqrt_d / n));
    }
  }
  __syncthreads();
  // 2. rotation to z = sqrt(d) * Pi x / n
  const float* rot = (is_key ? P.k_rot : P.v_rot) + (size_t)head * (P.kind == TQ_FWHT ? D : D * D);
  rotate_tile<D>(s, nv, P.kind, rot);
  // 3. codes, planes, residual
  const int j = tid;
  const bool wide = split && j < D / 2;
  const int bj = bits + (wide ? 1 : 0);         // bits of this coordinate
  const int nplanes = bits + (split ? 1 : 0);   // planes of the tile (warp-uniform)
  const float* tbj = wide ? s.tb_hi : s.tb;
  const float* cbj = wide ? s.cb_hi : s.cb;
  unsigned vm[TQ_MAX_BITS] = {0u, 0u, 0u, 0u};
  for (int v = 0; v < nv; ++v) {
    const float z = s.x[v][j];
    const int idx = bucketize(z, tbj, bj);
#pragma unroll
    for (int p = 0; p < TQ_MAX_BITS; ++p) {
      if (p < nplanes) {
        const unsigned b = p < bj ? plane_bit(idx, bj, p) : 0u;  // the top plane: first half only
        const unsigned w = __ballot_sync(0xffffffffu, b);
        if (lane == 0) s.codes[v][p][warp] = w;
        if (slot_of && slot_of[v] >= 0) vm[p] |= b << slot_of[v];
      }
    }
    if (is_key) {
      const float c = cbj[idx];
      // QJL: residual; EDEN / length-renormalized: z c (z and c share a sign, so the terms are >= 0)
      s.r[v][j] = (P.kqjl == TQ_KEY_EDEN || P.kqjl == TQ_KEY_RENORM) ? z * c : z - c;
    }
  }
  if (!is_key && slot_of) {
#pragma unroll
    for (int p = 0; p < TQ_MAX_BITS; ++p) s.vmask[p][j] = vm[p];
  }
  __syncthreads();
  if (!is_key) return;
  // 4. residual norm gamma = ||z - C|| / sqrt(d), or the key scale s from the sum of the r entries
  const bool scaled = P.kqjl == TQ_KEY_EDEN || P.kqjl == TQ_KEY_RENORM;
  if constexpr (ONE) {
    if (warp == 0) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float rv = s.r[0][e * 32 + lane];
        acc = scaled ? acc + rv : fmaf(rv, rv, acc);
      }
      acc = warp_sum_f(acc);
      if (lane == 0) {
        const float g = scaled ? (float)D / acc : sqrtf(acc) / sqrt_d;
        s.gam[0] = s.zero[0] ? 0.f : g;
      }
    }
  } else for (int v = warp; v < nv; v += D / 32) {
    double acc = 0.0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const double rv = s.r[v][e * 32 + lane];
      acc += scaled ? rv : rv * rv;
    }
    acc = warp_sum_d(acc);
    if (lane == 0) {
      const double g = scaled ? (double)D / acc : sqrt(acc) / (double)sqrt_d;
      s.gam[v] = s.zero[v] ? 0.f : (float)g;
    }
  }
  if (P.kqjl != TQ_KEY_QJL) {
    __syncthreads();
    return;
  }
  if (P.qjl_srht) {
    // 5. structured sketch S = H diag(sigma_S): signs of the fast transform of sigma_S * r,
    //    one warp per vector (coordinate e * 32 + lane in register e, word e of the signs)
    const float* sg = P.qjl_s + (size_t)head * D;
    for (int v = warp; v < nv; v += D / 32) {
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = s.r[v][e * 32 + lane] * __ldg(sg + e * 32 + lane);
      warp_wht<E>(a, lane);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const unsigned w = __ballot_sync(0xffffffffu, (s.zero[v] || a[e] >= 0.f) ? 1u : 0u);
        if (lane == 0) s.signs[v][e] = w;
      }
    }
    __syncthreads();
    return;
  }
  // 5. QJL signs of S r (r in z units; the sign is scale free)
  if constexpr (ONE) {
    // one vector: warp w takes rows 32 w .. 32 w + 31 of S, its lanes along a row (coalesced loads,
    // a warp sum a row) instead of a thread a row, sixteen rows of loads in flight
    const float* S0 = P.qjl_s + (size_t)head * D * D;
    constexpr int kRows = 16, kH = D / 128;  // rows of S a batch, float4 loads a lane and row
    unsigned mine = 0u;
#pragma unroll 1
    for (int r0 = 0; r0 < 32; r0 += kRows) {
      float4 p[kRows][kH];
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        const float4* srow = reinterpret_cast<const float4*>(S0 + (size_t)(32 * warp + r0 + rr) * D);
#pragma unroll
        for (int h = 0; h < kH; ++h) p[rr][h] = __ldg(srow + lane + 32 * h);
      }
      float a[kRows];
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        a[rr] = 0.f;
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          const float4 rv = *reinterpret_cast<const float4*>(&s.r[0][(lane + 32 * h) * 4]);
          const float4 q = p[rr][h];
          a[rr] = fmaf(q.x, rv.x, fmaf(q.y, rv.y, fmaf(q.z, rv.z, fmaf(q.w, rv.w, a[rr]))));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) a[rr] += __shfl_xor_sync(0xffffffffu, a[rr], o);
      }
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr)
        if (lane == r0 + rr && (s.zero[0] || a[rr] >= 0.f)) mine = 1u;
    }
    const unsigned w = __ballot_sync(0xffffffffu, mine);
    if (lane == 0) s.signs[0][warp] = w;
    __syncthreads();
    return;
  }
  const float4* row = reinterpret_cast<const float4*>(P.qjl_s + (size_t)head * D * D + (size_t)j * D);
  float acc[kTile];
#pragma unroll
  for (int v = 0; v < kTile; ++v) acc[v] = 0.f;
  // eight rows of S in flight: a decode-step append (one vector) waits on these loads alone
#pragma unroll 8
  for (int i4 = 0; i4 < D / 4; ++i4) {
    const float4 p = __ldg(row + i4);
#pragma unroll
    for (int v = 0; v < kTile; ++v) {
      if (v < nv) {
        const float4 rv = *reinterpret_cast<const float4*>(&s.r[v][i4 * 4]);
        acc[v] = fmaf(p.x, rv.x, acc[v]);
        acc[v] = fmaf(p.y, rv.y, acc[v]);
        acc[v] = fmaf(p.z, rv.z, acc[v]);
        acc[v] = fmaf(p.w, rv.w, acc[v]);
      }
    }
  }
  for (int v = 0; v < nv; ++v) {
    const unsigned b = (s.zero[v] || acc[v] >= 0.f) ? 1u : 0u;
    const unsigned w = __ballot_sync(0xffffffffu, b);
    if (lane == 0) s.signs[v][warp] = w;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ flat quantize

template <int D>
__global__ void __launch_bounds__(D) quantize_flat_kernel(const __grid_constant__ KParams P, const void* x,
                                                          int dtype, long long n_vec, int is_key,
                                                          uint32_t* codes, uint32_t* signs, float* norms,
                                                          float* rnorms) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<D>& s = *reinterpret_cast<TileSmem<D>*>(smem_raw);
  constexpr int E = D / 32;
  const int head = blockIdx.y;
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const int bits = is_key ? P.kb : P.vb;
  for (long long t0 = (long long)blockIdx.x * kTile; t0 < n_tok; t0 += (long long)gridDim.x * kTile) {
    int nv = 0;
    // tile = tokens t0..t0+15 of this head; vector n = t * hkv + head
    for (int v = 0; v < kTile; ++v) {
      const long long n = (t0 + v) * P.hkv + head;
      if (t0 + v < n_tok && n < n_vec) nv = v + 1;
    }
    for (int v = 0; v < nv; ++v) {
      const long long n = (t0 + v) * P.hkv + head;
      s.x[v][threadIdx.x] = threadIdx.x < P.dh ? load_elem(x, dtype, n * P.dh + threadIdx.x) : 0.f;  // zero-padded to D
    }
    __syncthreads();
    quantize_tile<D>(P, s, nv, head, is_key != 0, nullptr);
    // stores: record words are contiguous per vector
    // mixed-channel keys: the top plane's first d/64 words follow the full planes
    const int words = bits * E + ((is_key && P.ksplit) ? E / 2 : 0);
    for (int i = threadIdx.x; i < nv * words; i += D) {
      const int v = i / words, k = i % words;
      const long long n = (t0 + v) * P.hkv + head;
      codes[n * words + k] = s.codes[v][k / E][k % E];
    }
    if (is_key && P.kqjl == TQ_KEY_QJL) {
      for (int i = threadIdx.x; i < nv * E; i += D) {
        const int v = i / E, k = i % E;
        const long long n = (t0 + v) * P.hkv + head;
        signs[n * E + k] = s.signs[v][k];
      }
    }
    if (threadIdx.x < nv) {
      const long long n = (t0 + threadIdx.x) * P.hkv + head;
      norms[n] = s.norm[threadIdx.x];
      if (is_key && P.kqjl) rnorms[n] = s.gam[threadIdx.x];  // gamma or the scale
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------ page stores

__device__ __forceinline__ unsigned char* subblock(const KParams& P, const KCache& C, long long page, int head) {
  return C.pool + ((size_t)page * P.hkv + head) * (size_t)P.sub_bytes;
}

// Store the key part of vector v at (page, slot).
template <int D>
__device__ void store_key_slot(const KParams& P, const TileSmem<D>& s, unsigned char* sb, int v, int slot) {
  constexpr int E = D / 32;
  uint32_t* kc = reinterpret_cast<uint32_t*>(sb + P.off_kcodes);
  for (int i = threadIdx.x; i < P.kb * E; i += D) {
    const int p = i / E, w = i % E;
    kc[(p * kPage + slot) * E + w] = s.codes[v][p][w];
  }
  if (P.ksplit) {
    uint32_t* kx = reinterpret_cast<uint32_t*>(sb + P.off_kx);
    for (int w = threadIdx.x; w < E / 2; w += D) kx[slot * (E / 2) + w] = s.codes[v][P.kb][w];
  }
  if (P.kqjl == TQ_KEY_QJL) {
    uint32_t* ks = reinterpret_cast<uint32_t*>(sb + P.off_ksigns);
    for (int w = threadIdx.x; w < E; w += D) ks[slot * E + w] = s.signs[v][w];
  }
  if (threadIdx.x == 0) {
    if (P.knu8) sb[P.off_knorm + slot] = norm_u8_encode(s.norm[v], P);
    else reinterpret_cast<float*>(sb + P.off_knorm)[slot] = s.norm[v];
    if (P.kqjl) reinterpret_cast<float*>(sb + P.off_krnorm)[slot] = s.gam[v];
  }
}

// Value planes of the tile into one sub-block: mask = slots written by this
// tile (bits of s.vmask outside mask are zero).  full == true writes whole
// words; otherwise read-modify-write with atomics (other slots may be written
// concurrently by other CTAs).
template <int D>
__device__ void store_value_planes(const KParams& P, const TileSmem<D>& s, unsigned char* sb, unsigned mask,
                                   bool full) {
  const int j = threadIdx.x;
  uint16_t* vc16 = reinterpret_cast<uint16_t*>(sb + P.off_vcodes);
  for (int p = 0; p < P.vb; ++p) {
    const unsigned bits = s.vmask[p][j] & mask;
    if (full) {
      vc16[p * D + j] = (uint16_t)bits;
    } else {
      unsigned int* w32 = reinterpret_cast<unsigned int*>(vc16 + p * D + (j & ~1));
      const int sh = (j & 1) * 16;
      atomicAnd(w32, ~(mask << sh));
      atomicOr(w32, bits << sh);
    }
  }
}

// Value planes of one vector v into slot `slot` of a sub-block (atomic
// read-modify-write: other slots of the page may be written concurrently).
template <int D>
__device__ void store_value_slot(const KParams& P, const TileSmem<D>& s, unsigned char* sb, int v, int slot) {
  const int j = threadIdx.x;
  uint16_t* vc16 = reinterpret_cast<uint16_t*>(sb + P.off_vcodes);
  for (int p = 0; p < P.vb; ++p) {
    const unsigned bit = (s.codes[v][p][j >> 5] >> (j & 31)) & 1u;
    unsigned int* w32 = reinterpret_cast<unsigned int*>(vc16 + p * D + (j & ~1));
    const int sh = (j & 1) * 16 + slot;
    atomicAnd(w32, ~(1u << sh));
    atomicOr(w32, bit << sh);
  }
}

// ------------------------------------------------------------------ KIVI control arm

// [Design study] §Candidate key and value algorithms, arm 3: asymmetric
// min-max integer codes, keys per channel over a page's 16 tokens, values per
// token over the d channels; scale = float16((max - min) / (2^b - 1)) formed in
// float32, zero = float16(min), code = clamp(floor((x - zero) / scale + 1/2)).

__device__ __forceinline__ void kivi_scale_zero(float mn, float mx, int bits, __half& hs, __half& hz) {
  hs = __float2half_rn(__fdiv_rn(mx - mn, (float)((1 << bits) - 1)));
  hz = __float2half_rn(mn);
}

__device__ __forceinline__ uint32_t kivi_code(float x, float sf, float zf, int bits) {
  if (!(sf > 0.f)) return 0u;
  const float t = __fdiv_rn(x - zf, sf);
  return (uint32_t)fminf(fmaxf(floorf(t + 0.5f), 0.f), (float)((1 << bits) - 1));
}

// The packed word of the lanes sharing it (32 / bits consecutive lanes): code of
// lane l at bits (l mod (32 / bits)) * bits.
__device__ __forceinline__ uint32_t kivi_word(uint32_t c, int bits, int lane) {
  const int per = 32 / bits;
  uint32_t w = c << ((lane % per) * bits);
  for (int o = 1; o < per; o <<= 1) w |= __shfl_xor_sync(0xffffffffu, w, o);
  return w;
}

// One whole page (16 tokens of one head, s.x[0..15][0..d)) into its sub-block:
// the key half (is_key) or the value half.
template <int D>
__device__ void kivi_store_page(const KParams& P, TileSmem<D>& s, bool is_key, unsigned char* sb) {
  const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
  const int bits = is_key ? P.kb : P.vb;
  const int per = 32 / bits, wpt = D * bits / 32;
  uint32_t* codes = reinterpret_cast<uint32_t*>(sb + (is_key ? P.off_kcodes : P.off_vcodes));
  if (is_key) {
    float mn = s.x[0][j], mx = mn;
    for (int t = 1; t < kPage; ++t) {
      mn = fminf(mn, s.x[t][j]);
      mx = fmaxf(mx, s.x[t][j]);
    }
    __half hs, hz;
    kivi_scale_zero(mn, mx, bits, hs, hz);
    reinterpret_cast<__half*>(sb + P.off_kscale)[j] = hs;
    reinterpret_cast<__half*>(sb + P.off_kzero)[j] = hz;
    const float sf = __half2float(hs), zf = __half2float(hz);
    for (int t = 0; t < kPage; ++t) {
      const uint32_t w = kivi_word(kivi_code(s.x[t][j], sf, zf, bits), bits, lane);
      if (lane % per == 0) codes[t * wpt + j / per] = w;
    }
  } else {
    for (int t = warp; t < kPage; t += D / 32) {  // warp w: tokens w, w + d/32, ...
      float mn = INFINITY, mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) {
        const float x = s.x[t][e * 32 + lane];
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (lane == 0) {
        __half hs, hz;
        kivi_scale_zero(mn, mx, bits, hs, hz);
        reinterpret_cast<__half*>(sb + P.off_vscale)[t] = hs;
        reinterpret_cast<__half*>(sb + P.off_vzero)[t] = hz;
        s.norm[t] = __half2float(hs);
        s.gam[t] = __half2float(hz);
      }
    }
    __syncthreads();
    for (int t = 0; t < kPage; ++t) {
      const uint32_t w = kivi_word(kivi_code(s.x[t][j], s.norm[t], s.gam[t], bits), bits, lane);
      if (lane % per == 0) codes[t * wpt + j / per] = w;
    }
  }
}

// ------------------------------------------------------------------ append: direct slots

// Direct slots.  With slot_mapping: token t of the input goes to pool slot slot_mapping[t].
// Without (prefill of whole sequences): token i = b n_c + p is position p of sequence b, read
// from input row b seq_tok + p and stored in page block_table[b][p / 16], slot p % 16.
template <int D>
__global__ void __launch_bounds__(D) append_direct_kernel(const __grid_constant__ KParams P,
                                                          const __grid_constant__ KCache C, const void* k,
                                                          const void* v, int dtype, long long n_tok,
                                                          const long long* slot_mapping, int seq_tok, int n_c) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<D>& s = *reinterpret_cast<TileSmem<D>*>(smem_raw);
  __shared__ int slot_of[kTile];
  __shared__ long long page_of[kTile];
  __shared__ long long row_of[kTile];
  __shared__ int same_page;
  const int head = blockIdx.y;
  const bool is_key = blockIdx.z == 0;
  const void* x = is_key ? k : v;
  for (long long t0 = (long long)blockIdx.x * kTile; t0 < n_tok; t0 += (long long)gridDim.x * kTile) {
    const int nv = (int)min((long long)kTile, n_tok - t0);
    if (threadIdx.x < kTile) {
      long long pg = -1;
      int sl = 0;
      long long row = t0 + threadIdx.x;
      if (threadIdx.x < nv) {
        long long sm = -1;
        if (slot_mapping) {
          sm = slot_mapping[t0 + threadIdx.x];
        } else {
          const long long i = t0 + threadIdx.x;
          const long long bq = i / n_c;
          const int pos = (int)(i - bq * n_c);
          row = bq * seq_tok + pos;
          if (pos / kPage < C.max_pages) {
            const long long pid = C.block_table[(size_t)bq * C.max_pages + pos / kPage];
            sm = pid >= 0 ? pid * kPage + pos % kPage : -1;
            if (pid < 0) atomicOr(&g_quant_err, TQ_DEVERR_SLOT);
          } else {
            atomicOr(&g_quant_err, TQ_DEVERR_SEQ_LEN);
          }
        }
        if (sm >= 0) {
          pg = sm / kPage;
          sl = (int)(sm % kPage);
          if (pg >= C.n_pages) {
            atomicOr(&g_quant_err, TQ_DEVERR_SLOT);
            pg = -1;
          }
        }
      }
      page_of[threadIdx.x] = pg;
      slot_of[threadIdx.x] = pg >= 0 ? sl : -1;
      row_of[threadIdx.x] = row;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      long long first = -1;
      int same = 1;
      for (int i = 0; i < nv; ++i) {
        if (page_of[i] < 0) continue;
        if (first < 0) first = page_of[i];
        else if (page_of[i] != first) same = 0;
      }
      same_page = same;
    }
    for (int i = 0; i < nv; ++i) {
      const long long n = row_of[i] * P.hkv + head;
      s.x[i][threadIdx.x] =
          (page_of[i] >= 0 && threadIdx.x < P.dh) ? load_elem(x, dtype, n * P.dh + threadIdx.x) : 0.f;
    }
    __syncthreads();
    if (P.kivi) {
      // whole pages only: the tile's 16 tokens fill slots 0..15 of one page in order
      bool whole = nv == kTile && same_page && page_of[0] >= 0;
      for (int i = 0; i < nv && whole; ++i) whole = slot_of[i] == i;
      if (whole) kivi_store_page<D>(P, s, is_key, subblock(P, C, page_of[0], head));
      else if (threadIdx.x == 0) atomicOr(&g_quant_err, TQ_DEVERR_SLOT);
      __syncthreads();
      continue;
    }
    quantize_tile<D>(P, s, nv, head, is_key, slot_of);
    if (is_key) {
      for (int i = 0; i < nv; ++i)
        if (page_of[i] >= 0) store_key_slot<D>(P, s, subblock(P, C, page_of[i], head), i, slot_of[i]);
    } else {
      if (same_page) {
        unsigned mask = 0;
        long long pg = -1;
        for (int i = 0; i < nv; ++i)
          if (page_of[i] >= 0) {
            mask |= 1u << slot_of[i];
            pg = page_of[i];
          }
        if (pg >= 0) {
          unsigned char* sb = subblock(P, C, pg, head);
          store_value_planes<D>(P, s, sb, mask, mask == 0xFFFFu);
        }
      } else {
        for (int i = 0; i < nv; ++i)
          if (page_of[i] >= 0) store_value_slot<D>(P, s, subblock(P, C, page_of[i], head), i, slot_of[i]);
      }
      if (threadIdx.x < nv && page_of[threadIdx.x] >= 0)
        reinterpret_cast<float*>(subblock(P, C, page_of[threadIdx.x], head) + P.off_vnorm)[slot_of[threadIdx.x]] =
            s.norm[threadIdx.x];
    }
    __syncthreads();
  }
}

}  // namespace tq

#include "tq_quantize256.cuh"

namespace tq {

// ------------------------------------------------------------------ append: decode step

// grid (batch, hkv, 2): blockIdx.z = 0 keys, 1 values.  Reads the counters;
// append_counters_kernel advances them afterwards (stream order).
template <int D>
__global__ void __launch_bounds__(D) append_step_kernel(const __grid_constant__ KParams P,
                                                        const __grid_constant__ KCache C, const void* k,
                                                        const void* v, int dtype) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<D>& s = *reinterpret_cast<TileSmem<D>*>(smem_raw);
  __shared__ int slot_of[kTile];
  const int b = blockIdx.x, head = blockIdx.y;
  const bool is_key = blockIdx.z == 0;
  const void* x = is_key ? k : v;
  const long long src = ((long long)b * P.hkv + head) * P.dh;
  const bool in_head = threadIdx.x < P.dh;  // coordinates >= dh are the zero padding
  // no window: every step quantizes its vector, so its load and (keys) the head's sketch rows toward
  // L2 are issued before the counters and the page lookup they would otherwise wait behind
  float x0 = 0.f;
  if (P.window == 0 && !P.kivi) {
    if (in_head) x0 = load_elem(x, dtype, src + threadIdx.x);
    if (is_key && P.kqjl == TQ_KEY_QJL && !P.qjl_srht) {
      const char* S0 = reinterpret_cast<const char*>(P.qjl_s + (size_t)head * D * D);
      for (int off = threadIdx.x * 128; off < D * D * (int)sizeof(float); off += D * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(S0 + off));
    }
  }
  const int T = C.seq_len[b];
  const int nc = C.n_compressed[b];
  if (P.window > 0) {
    __half* ring = (is_key ? C.win_k : C.win_v) + (((size_t)b * P.hkv + head) * C.ring) * D;
    if (T - nc < 0 || T - nc >= P.window + kPage) {
      if (threadIdx.x == 0) atomicOr(&g_quant_err, TQ_DEVERR_SEQ_LEN);
      return;
    }
    ring[(size_t)(T % C.ring) * D + threadIdx.x] = __float2half_rn(in_head ? load_elem(x, dtype, src + threadIdx.x) : 0.f);
    if (T + 1 - nc != P.window + kPage) return;
    // flush the oldest 16 window tokens into page nc / 16
    const int pidx = nc / kPage;
    long long page = -1;
    if (pidx < C.max_pages) page = C.block_table[(size_t)b * C.max_pages + pidx];
    if (page < 0 || page >= C.n_pages) {
      if (threadIdx.x == 0) atomicOr(&g_quant_err, pidx < C.max_pages ? TQ_DEVERR_PAGE_INDEX : TQ_DEVERR_SEQ_LEN);
      return;
    }
    for (int i = 0; i < kPage; ++i)
      s.x[i][threadIdx.x] = __half2float(ring[(size_t)((nc + i) % C.ring) * D + threadIdx.x]);
    if (threadIdx.x < kTile) slot_of[threadIdx.x] = threadIdx.x;
    __syncthreads();
    if (P.kivi) {
      kivi_store_page<D>(P, s, is_key, subblock(P, C, page, head));
      return;
    }
    quantize_tile<D>(P, s, kPage, head, is_key, slot_of);
    unsigned char* sb = subblock(P, C, page, head);
    if (is_key) {
      for (int i = 0; i < kPage; ++i) store_key_slot<D>(P, s, sb, i, i);
    } else {
      store_value_planes<D>(P, s, sb, 0xFFFFu, true);
      if (threadIdx.x < kPage) reinterpret_cast<float*>(sb + P.off_vnorm)[threadIdx.x] = s.norm[threadIdx.x];
    }
  } else {
    if (P.kivi) {  // the KIVI arm needs a window (checked on the host)
      if (threadIdx.x == 0) atomicOr(&g_quant_err, TQ_DEVERR_SEQ_LEN);
      return;
    }
    const int pidx = T / kPage, slot = T % kPage;
    long long page = -1;
    if (T >= 0 && pidx < C.max_pages) page = C.block_table[(size_t)b * C.max_pages + pidx];
    if (page < 0 || page >= C.n_pages) {
      if (threadIdx.x == 0)
        atomicOr(&g_quant_err, (T >= 0 && pidx < C.max_pages) ? TQ_DEVERR_PAGE_INDEX : TQ_DEVERR_SEQ_LEN);
      return;
    }
    s.x[0][threadIdx.x] = x0;
    if (threadIdx.x == 0) slot_of[0] = slot;
    __syncthreads();
    quantize_tile<D, true>(P, s, 1, head, is_key, slot_of);
    unsigned char* sb = subblock(P, C, page, head);
    if (is_key) {
      store_key_slot<D>(P, s, sb, 0, slot);
    } else {
      store_value_slot<D>(P, s, sb, 0, slot);
      if (threadIdx.x == 0) reinterpret_cast<float*>(sb + P.off_vnorm)[slot] = s.norm[0];
    }
  }
}

// Prefill of whole sequences: positions n_c .. seq_tok - 1 of every (sequence, kv head) into the
// float16 window ring (slot p mod ring, rows of d with a zero tail past head_dim).  grid (batch, hkv, 2).
template <int D>
__global__ void __launch_bounds__(D) prefill_window_kernel(const __grid_constant__ KParams P,
                                                           const __grid_constant__ KCache C, const void* k,
                                                           const void* v, int dtype, int seq_tok, int n_c) {
  const int b = blockIdx.x, head = blockIdx.y, j = threadIdx.x;
  const bool is_key = blockIdx.z == 0;
  const void* x = is_key ? k : v;
  __half* ring = (is_key ? C.win_k : C.win_v) + (((size_t)b * P.hkv + head) * C.ring) * D;
  for (int p = n_c; p < seq_tok; ++p) {
    const long long n = ((long long)b * seq_tok + p) * P.hkv + head;
    ring[(size_t)(p % C.ring) * D + j] = __float2half_rn(j < P.dh ? load_elem(x, dtype, n * P.dh + j) : 0.f);
  }
}

__global__ void prefill_counters_kernel(const __grid_constant__ KCache C, int seq_tok, int n_c) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= C.batch) return;
  C.seq_len[b] = seq_tok;
  C.n_compressed[b] = n_c;
}

__global__ void append_counters_kernel(const __grid_constant__ KCache C, int window) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= C.batch) return;
  const int T = C.seq_len[b];
  int nc = C.n_compressed[b];
  if (window > 0) {
    if (T - nc < 0 || T - nc >= window + kPage) return;  // flagged by the step kernel
    if (T + 1 - nc == window + kPage) nc += kPage;
  } else {
    if (T / kPage >= C.max_pages) return;
    nc = T + 1;
  }
  C.seq_len[b] = T + 1;
  C.n_compressed[b] = nc;
}

// ------------------------------------------------------------------ launchers

template <int D>
static size_t tile_smem() {
  return sizeof(TileSmem<D>);
}

template <int D>
static cudaError_t launch_quantize_flat_d(const KParams& P, const void* x, int dtype, long long n_vec, bool is_key,
                                          uint32_t* codes, uint32_t* signs, float* norms, float* rnorms,
                                          cudaStream_t st) {
  const size_t sm = tile_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(quantize_flat_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  long long tiles = (n_tok + kTile - 1) / kTile;
  const int gx = (int)std::min<long long>(tiles, 65535);
  dim3 grid(gx, P.hkv);
  quantize_flat_kernel<D><<<grid, D, sm, st>>>(P, x, dtype, n_vec, is_key ? 1 : 0, codes, signs, norms, rnorms);
  return cudaGetLastError();
}

// Codebook tables with c[half + m] = -c[half - 1 - m], a zero middle boundary,
// antisymmetric and strictly increasing boundaries (tq_build_codebook's tables).
static bool antisymmetric(const float* c, const float* t, int bits) {
  const int half = 1 << (bits - 1);
  if (t[half - 1] != 0.f) return false;
  for (int m = 0; m < half; ++m)
    if (c[half + m] != -c[half - 1 - m]) return false;
  for (int k = 1; k < half; ++k)
    if (t[half - 1 + k] != -t[half - 1 - k]) return false;
  for (int k = half - 1; k + 1 < 2 * half - 1; ++k)
    if (!(t[k] < t[k + 1])) return false;
  return true;
}

// Scale J of the code cell table (wq::code_cell): the smallest J <= kLutMaxJ for which
// the 2^bits - 1 boundaries fall in distinct cells, else -1.
static int code_lut_scale(const float* t, int bits) {
  const int nb = (1 << bits) - 1;
  for (int J = 0; J <= wq::kLutMaxJ; ++J) {
    const float sc = (float)(32 << J);
    bool ok = true;
    for (int k = 0; k + 1 < nb && ok; ++k) ok = wq::code_cell(t[k], sc) < wq::code_cell(t[k + 1], sc);
    if (ok) return J;
  }
  return -1;
}

template <int BITS, bool DENSE, int MODE>
static cudaError_t launch_quantize_warp(const KParams& P, const KCache& C, const void* x, long long n_vec,
                                        bool is_key, uint32_t* codes, uint32_t* signs, float* norms, float* rnorms,
                                        cudaStream_t st) {
  constexpr int warps = wq::warps_for(DENSE);
  auto kern = wq::quantize_warp_kernel<BITS, DENSE, MODE>;
  const int J = code_lut_scale(is_key ? P.kt : P.vt, BITS);
  const size_t sm = wq::smem_bytes(DENSE) + wq::lut_bytes(J, true);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  int occ = 0, dev = 0, sms = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, 32 * warps, sm)) != cudaSuccess) return e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 15) / 16;
  if (n_tiles == 0) return cudaSuccess;
  long long gx = std::max(1LL, (long long)std::max(occ, 1) * sms / P.hkv);
  // bulk: adjacent tiles per CTA; a decode-step append interleaves its tiles over as many CTAs
  gx = std::min(gx, MODE == wq::kStep ? n_tiles : (n_tiles + warps - 1) / warps);
  dim3 grid((int)std::min(gx, 65535LL), P.hkv);
  kern<<<grid, 32 * warps, sm, st>>>(P, C, reinterpret_cast<const __nv_bfloat16*>(x), n_vec, is_key ? 1 : 0,
                                      codes, signs, norms, rnorms, J);
  return cudaGetLastError();
}

template <bool DENSE, int MODE>
static cudaError_t launch_quantize_warp_bits(int bits, const KParams& P, const KCache& C, const void* x,
                                             long long n_vec, bool is_key, uint32_t* codes, uint32_t* signs,
                                             float* norms, float* rnorms, cudaStream_t st) {
  switch (bits) {
    case 1: return launch_quantize_warp<1, DENSE, MODE>(P, C, x, n_vec, is_key, codes, signs, norms, rnorms, st);
    case 2: return launch_quantize_warp<2, DENSE, MODE>(P, C, x, n_vec, is_key, codes, signs, norms, rnorms, st);
    case 3: return launch_quantize_warp<3, DENSE, MODE>(P, C, x, n_vec, is_key, codes, signs, norms, rnorms, st);
    default: return launch_quantize_warp<4, DENSE, MODE>(P, C, x, n_vec, is_key, codes, signs, norms, rnorms, st);
  }
}

// Tensor-core path: d = 128, bf16, 16-byte aligned input, antisymmetric tables.
static bool warp_path_ok(const KParams& P, const void* x, int dtype, bool is_key, long long n_vec) {
  // mixed-channel keys and byte norms: CUDA-core tiles
  if (is_key && (P.ksplit || P.knu8)) return false;
  if (P.kivi) return false;
  const bool sym = is_key ? antisymmetric(P.kc, P.kt, P.kb) : antisymmetric(P.vc, P.vt, P.vb);
  const int J = is_key ? code_lut_scale(P.kt, P.kb) : code_lut_scale(P.vt, P.vb);
  // the dense key kernel's shared memory (operand tiles and Pi limbs) leaves room for J <= 2
  const bool fits = J >= 0 && !(is_key && P.kqjl == TQ_KEY_QJL && P.kind != TQ_FWHT && J > 2);
  return P.d == 128 && dtype == TQ_BF16 && sym && fits && ((uintptr_t)x & 15) == 0 && n_vec < (1LL << 32);
}

template <int BITS, bool DENSE, int MODE>
static cudaError_t launch_quantize_keys_tc(const KParams& P, const KCache& C, const void* x, long long n_vec,
                                           uint32_t* codes, uint32_t* signs, float* norms, float* rnorms,
                                           cudaStream_t st) {
  auto kern = wq::quantize_keys_tc_kernel<BITS, DENSE, MODE>;
  const int J = code_lut_scale(P.kt, BITS);
  const size_t sm = wq::tc_smem_bytes(DENSE) + wq::lut_bytes(J, false);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 15) / 16;
  if (n_tiles == 0) return cudaSuccess;
  // warp tiles a CTA pass: all 8 for bulk calls; a decode-step append spreads its tiles over
  // the SMs (one CTA per SM for the shared memory) when it has fewer than 8 a CTA
  int tp = wq::kTcWarps;
  if (MODE == wq::kStep)
    tp = (int)std::min<long long>(wq::kTcWarps, std::max<long long>(1, (n_tiles * P.hkv + sms - 1) / sms));
  const long long n_ct = (n_tiles + tp - 1) / tp;
  long long gx = std::max(1LL, (long long)sms / P.hkv);  // one CTA per SM (shared memory)
  gx = std::min(gx, n_ct);
  dim3 grid((int)std::min(gx, 65535LL), P.hkv);
  kern<<<grid, 32 * wq::kTcWarps, sm, st>>>(P, C, reinterpret_cast<const __nv_bfloat16*>(x), n_vec, codes, signs,
                                            norms, rnorms, J, tp);
  return cudaGetLastError();
}

template <bool DENSE, int MODE>
static cudaError_t launch_quantize_keys_tc_bits(int bits, const KParams& P, const KCache& C, const void* x,
                                                long long n_vec, uint32_t* codes, uint32_t* signs, float* norms,
                                                float* rnorms, cudaStream_t st) {
  switch (bits) {
    case 1: return launch_quantize_keys_tc<1, DENSE, MODE>(P, C, x, n_vec, codes, signs, norms, rnorms, st);
    case 2: return launch_quantize_keys_tc<2, DENSE, MODE>(P, C, x, n_vec, codes, signs, norms, rnorms, st);
    case 3: return launch_quantize_keys_tc<3, DENSE, MODE>(P, C, x, n_vec, codes, signs, norms, rnorms, st);
    default: return launch_quantize_keys_tc<4, DENSE, MODE>(P, C, x, n_vec, codes, signs, norms, rnorms, st);
  }
}

template <int MODE>
static cudaError_t launch_quantize_warp_role(const KParams& P, const KCache& C, const void* x, long long n_vec,
                                             bool is_key, uint32_t* codes, uint32_t* signs, float* norms,
                                             float* rnorms, cudaStream_t st) {
  const bool qjl = is_key && P.kqjl == TQ_KEY_QJL;
  const int bits = is_key ? P.kb : P.vb;
  if (qjl)  // keys with the sketch: tcgen05 for S r (record indices fit 32 bits)
    return P.kind == TQ_FWHT
               ? launch_quantize_keys_tc_bits<false, MODE>(bits, P, C, x, n_vec, codes, signs, norms, rnorms, st)
               : launch_quantize_keys_tc_bits<true, MODE>(bits, P, C, x, n_vec, codes, signs, norms, rnorms, st);
  if (P.kind == TQ_FWHT)
    return launch_quantize_warp_bits<false, MODE>(bits, P, C, x, n_vec, is_key, codes, signs, norms, rnorms, st);
  return launch_quantize_warp_bits<true, MODE>(bits, P, C, x, n_vec, is_key, codes, signs, norms, rnorms, st);
}

// FWHT keys with the QJL sketch, both products on tcgen05 (wq::quantize_bt_kernel).
template <int BITS>
static cudaError_t launch_quantize_bt(const KParams& P, const void* x, long long n_vec, uint32_t* codes,
                                      uint32_t* signs, float* norms, float* rnorms, int J, cudaStream_t st) {
  auto kern = wq::quantize_bt_kernel<BITS>;
  const size_t sm = wq::bt_smem_bytes(J);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 127) / 128;
  if (n_tiles == 0) return cudaSuccess;
  long long gx = std::max(1LL, (long long)sms / P.hkv);  // one CTA (two groups) per SM
  gx = std::min(gx, (n_tiles + 1) / 2);
  dim3 grid((int)std::min(gx, 65535LL), P.hkv);
  kern<<<grid, wq::kBtThreads, sm, st>>>(P, reinterpret_cast<const __nv_bfloat16*>(x), n_vec, codes, signs, norms,
                                        rnorms, J);
  return cudaGetLastError();
}

// Keys with the QJL sketch, FWHT: the tcgen05 kernel, when its shared memory (the operand
// tiles leave room for cell tables with J <= 1) fits the device's opt-in limit.
static bool bt_path_ok(const KParams& P, bool is_key) {
  if (!is_key || P.kqjl != TQ_KEY_QJL || P.kind != TQ_FWHT || P.dh > 128 || P.dh % 8 != 0) return false;
  const int J = code_lut_scale(P.kt, P.kb);
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  return J >= 0 && wq::bt_smem_bytes(J) <= (size_t)optin;
}

// Dense Pi, values and keys without the sketch: the rotation on tcgen05 (wq::quantize_bv_kernel).
template <int BITS, int ROLE>
static cudaError_t launch_quantize_bv(const KParams& P, const void* x, long long n_vec, uint32_t* codes,
                                      float* norms, float* rnorms, int J, cudaStream_t st) {
  auto kern = wq::quantize_bv_kernel<BITS, ROLE>;
  const size_t sm = wq::bv_smem_bytes(J);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 127) / 128;
  if (n_tiles == 0) return cudaSuccess;
  long long gx = std::max(1LL, (long long)sms / P.hkv);  // one CTA (four groups) per SM
  gx = std::min(gx, (n_tiles + wq::kBvGroups - 1) / wq::kBvGroups);
  dim3 grid((int)std::min(gx, 65535LL), P.hkv);
  kern<<<grid, wq::kBtThreads, sm, st>>>(P, reinterpret_cast<const __nv_bfloat16*>(x), n_vec, codes, norms, rnorms,
                                        J);
  return cudaGetLastError();
}

template <int ROLE>
static cudaError_t launch_quantize_bv_bits(int bits, const KParams& P, const void* x, long long n_vec,
                                           uint32_t* codes, float* norms, float* rnorms, int J, cudaStream_t st) {
  switch (bits) {
    case 1: return launch_quantize_bv<1, ROLE>(P, x, n_vec, codes, norms, rnorms, J, st);
    case 2: return launch_quantize_bv<2, ROLE>(P, x, n_vec, codes, norms, rnorms, J, st);
    case 3: return launch_quantize_bv<3, ROLE>(P, x, n_vec, codes, norms, rnorms, J, st);
    default: return launch_quantize_bv<4, ROLE>(P, x, n_vec, codes, norms, rnorms, J, st);
  }
}

// Dense Pi without the sketch: the tcgen05 kernel when its shared memory fits.
static bool bv_path_ok(const KParams& P, bool is_key) {
  if (P.kind == TQ_FWHT || (is_key && P.kqjl == TQ_KEY_QJL) || P.dh > 128 || P.dh % 8 != 0) return false;
  const int J = is_key ? code_lut_scale(P.kt, P.kb) : code_lut_scale(P.vt, P.vb);
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  return J >= 0 && wq::bv_smem_bytes(J) <= (size_t)optin;
}

cudaError_t launch_quantize_flat(const KParams& P, const void* x, int dtype, long long n_vec, bool is_key,
                                 uint32_t* codes, uint32_t* signs, float* norms, float* rnorms, cudaStream_t st) {
  if (warp_path_ok(P, x, dtype, is_key, n_vec) && bt_path_ok(P, is_key)) {
    const int J = code_lut_scale(P.kt, P.kb);
    switch (P.kb) {
      case 1: return launch_quantize_bt<1>(P, x, n_vec, codes, signs, norms, rnorms, J, st);
      case 2: return launch_quantize_bt<2>(P, x, n_vec, codes, signs, norms, rnorms, J, st);
      case 3: return launch_quantize_bt<3>(P, x, n_vec, codes, signs, norms, rnorms, J, st);
      default: return launch_quantize_bt<4>(P, x, n_vec, codes, signs, norms, rnorms, J, st);
    }
  }
  if (warp_path_ok(P, x, dtype, is_key, n_vec) && bv_path_ok(P, is_key)) {
    const int bits = is_key ? P.kb : P.vb;
    const int J = code_lut_scale(is_key ? P.kt : P.vt, bits);
    if (!is_key) return launch_quantize_bv_bits<0>(bits, P, x, n_vec, codes, norms, rnorms, J, st);
    if (P.kqjl == TQ_KEY_EDEN || P.kqjl == TQ_KEY_RENORM)
      return launch_quantize_bv_bits<2>(bits, P, x, n_vec, codes, norms, rnorms, J, st);
    return launch_quantize_bv_bits<3>(bits, P, x, n_vec, codes, norms, rnorms, J, st);
  }
  if (warp_path_ok(P, x, dtype, is_key, n_vec))
    return launch_quantize_warp_role<wq::kFlat>(P, KCache{}, x, n_vec, is_key, codes, signs, norms, rnorms, st);
  if (P.d == 128) return launch_quantize_flat_d<128>(P, x, dtype, n_vec, is_key, codes, signs, norms, rnorms, st);
  return launch_quantize_flat_d<256>(P, x, dtype, n_vec, is_key, codes, signs, norms, rnorms, st);
}

// d = 256 direct slots through q256::direct256_kernel (FWHT kind, uniform key rate, float norms).
static bool direct256_ok(const KParams& P) {
  return P.d == 256 && P.kind == TQ_FWHT && !P.kivi && !P.ksplit && !P.knu8 && antisymmetric(P.kc, P.kt, P.kb) &&
         antisymmetric(P.vc, P.vt, P.vb) && code_lut_scale(P.kt, P.kb) >= 0 && code_lut_scale(P.vt, P.vb) >= 0;
}

template <bool KEY, int SK>
static cudaError_t launch_direct256_role(const KParams& P, const KCache& C, const void* x, int dtype, long long n_tok,
                                         const long long* slots, int seq_tok, int n_c, cudaStream_t st) {
  auto kern = q256::direct256_kernel<KEY, SK>;
  const int J = KEY ? code_lut_scale(P.kt, P.kb) : code_lut_scale(P.vt, P.vb);
  const size_t sm = q256::smem_bytes(SK == 1) + wq::lut_bytes(J, false);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const long long tiles = (n_tok + q256::TILE - 1) / q256::TILE;
  const int per_sm = (KEY && SK == 1) ? 1 : 2;  // the sketch stages S in 128 KB of shared memory
  const long long gx = std::min<long long>(std::max(1, per_sm * sms / std::max(1, P.hkv)), tiles);
  kern<<<dim3((unsigned)std::max<long long>(gx, 1), P.hkv), q256::NT, sm, st>>>(P, C, x, dtype, n_tok, slots, seq_tok, n_c,
                                                                               J);
  return cudaGetLastError();
}

static cudaError_t launch_direct256_values(const KParams& P, const KCache& C, const void* v, int dtype, long long n_tok,
                                           const long long* slots, int seq_tok, int n_c, cudaStream_t st) {
  const int J = code_lut_scale(P.vt, P.vb);
  const size_t sm = wq::lut_bytes(J, true);
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q256::direct256_values_kernel, 32 * q256::VNW, sm)) !=
      cudaSuccess)
    return e;
  const long long groups = slots ? (n_tok + 15) / 16 : (n_c > 0 ? n_tok / n_c : 0) * ((n_c + kPage - 1) / kPage);
  const long long ctas = (groups + q256::VNW - 1) / q256::VNW;
  const long long gx = std::min<long long>(std::max(1, std::max(1, per_sm) * sms / std::max(1, P.hkv)), ctas);
  q256::direct256_values_kernel<<<dim3((unsigned)std::max<long long>(gx, 1), P.hkv), 32 * q256::VNW, sm, st>>>(
      P, C, v, dtype, n_tok, slots, seq_tok, n_c, J);
  return cudaGetLastError();
}

static cudaError_t launch_direct256(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                    long long n_tok, const long long* slots, int seq_tok, int n_c, cudaStream_t st) {
  cudaError_t e;
  if (P.kqjl == TQ_KEY_QJL)
    e = P.qjl_srht ? launch_direct256_role<true, 2>(P, C, k, dtype, n_tok, slots, seq_tok, n_c, st)
                   : launch_direct256_role<true, 1>(P, C, k, dtype, n_tok, slots, seq_tok, n_c, st);
  else
    e = launch_direct256_role<true, 0>(P, C, k, dtype, n_tok, slots, seq_tok, n_c, st);
  if (e != cudaSuccess) return e;
  return launch_direct256_values(P, C, v, dtype, n_tok, slots, seq_tok, n_c, st);
}

template <int D>
static cudaError_t launch_append_direct_d(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                          long long n_tok, const long long* slots, int seq_tok, int n_c,
                                          cudaStream_t st) {
  const size_t sm = tile_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(append_direct_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  const long long tiles = (n_tok + kTile - 1) / kTile;
  dim3 grid((int)std::min<long long>(tiles, 65535), P.hkv, 2);
  append_direct_kernel<D><<<grid, D, sm, st>>>(P, C, k, v, dtype, n_tok, slots, seq_tok, n_c);
  return cudaGetLastError();
}

cudaError_t launch_append_direct(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                 long long n_tok, const long long* slots, cudaStream_t st) {
  if (P.d == 128) return launch_append_direct_d<128>(P, C, k, v, dtype, n_tok, slots, 0, 1, st);
  if (direct256_ok(P)) return launch_direct256(P, C, k, v, dtype, n_tok, slots, 0, 1, st);
  return launch_append_direct_d<256>(P, C, k, v, dtype, n_tok, slots, 0, 1, st);
}

template <int D>
static cudaError_t launch_prefill_cache_d(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                          int seq_tok, int n_c, cudaStream_t st) {
  cudaError_t e = cudaSuccess;
  if (n_c > 0) {
    e = direct256_ok(P) ? launch_direct256(P, C, k, v, dtype, (long long)C.batch * n_c, nullptr, seq_tok, n_c, st)
                        : launch_append_direct_d<D>(P, C, k, v, dtype, (long long)C.batch * n_c, nullptr, seq_tok, n_c, st);
    if (e != cudaSuccess) return e;
  }
  if (seq_tok > n_c) {
    prefill_window_kernel<D><<<dim3(C.batch, P.hkv, 2), D, 0, st>>>(P, C, k, v, dtype, seq_tok, n_c);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  prefill_counters_kernel<<<(C.batch + 127) / 128, 128, 0, st>>>(C, seq_tok, n_c);
  return cudaGetLastError();
}

cudaError_t launch_prefill_cache(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                 int seq_tok, int n_c, cudaStream_t st) {
  if (P.d == 128) return launch_prefill_cache_d<128>(P, C, k, v, dtype, seq_tok, n_c, st);
  return launch_prefill_cache_d<256>(P, C, k, v, dtype, seq_tok, n_c, st);
}

template <int D>
static cudaError_t launch_append_step_d(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                                        cudaStream_t st) {
  if (P.window == 0 && warp_path_ok(P, k, dtype, true, (long long)C.batch * P.hkv) &&
      warp_path_ok(P, v, dtype, false, (long long)C.batch * P.hkv)) {
    // one sequence per row of the warp tiles: keys, values, then the counters
    const long long n_vec = (long long)C.batch * P.hkv;
    cudaError_t e = launch_quantize_warp_role<wq::kStep>(P, C, k, n_vec, true, nullptr, nullptr, nullptr, nullptr, st);
    if (e != cudaSuccess) return e;
    e = launch_quantize_warp_role<wq::kStep>(P, C, v, n_vec, false, nullptr, nullptr, nullptr, nullptr, st);
    if (e != cudaSuccess) return e;
    append_counters_kernel<<<(C.batch + 127) / 128, 128, 0, st>>>(C, P.window);
    return cudaGetLastError();
  }
  const size_t sm = tile_smem<D>();
  cudaError_t e = cudaFuncSetAttribute(append_step_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
  if (e != cudaSuccess) return e;
  dim3 grid(C.batch, P.hkv, 2);
  append_step_kernel<D><<<grid, D, sm, st>>>(P, C, k, v, dtype);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  append_counters_kernel<<<(C.batch + 127) / 128, 128, 0, st>>>(C, P.window);
  return cudaGetLastError();
}

cudaError_t launch_append_step(const KParams& P, const KCache& C, const void* k, const void* v, int dtype,
                               cudaStream_t st) {
  if (P.d == 128) return launch_append_step_d<128>(P, C, k, v, dtype, st);
  return launch_append_step_d<256>(P, C, k, v, dtype, st);
}

cudaError_t read_clear_quant_error(unsigned* bits) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_quant_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_quant_err, &zero, sizeof(unsigned));
}

}  // namespace tq
