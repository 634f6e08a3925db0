// Device-side definitions shared by the kernels of libtq (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tq.h"

namespace tq {

constexpr int kPage = 16;      // tokens per page
constexpr int kTile = 16;      // vectors per quantize tile
constexpr float kZeroNorm = 1e-7f;

// Kernel-side copy of tq_layer_params plus the derived page layout.
struct KParams {
  int d, hkv, hq, G, window, kb, kqjl, vb, kind;
  int dh;                              // length of the caller's vectors (<= d; zero-padded to d)
  const float* k_rot;
  const float* v_rot;
  const float* qjl_s;
  int qjl_srht;                        // qjl_s holds the signs of S = H diag(sigma_S)
  float kc[16], kt[16], vc[16], vt[16];
  // Walsh-plane coefficients: a code (sign s, magnitude bits m) has centroid
  // s * sum_S a_S * prod_{i in S} (1 - 2 m_i); plane S has bit s ^ parity(m & S).
  float akw[8], avw[8];
  // mixed-channel key rate: coordinates < d/2 take kb + 1 bits with the kc_hi / kt_hi book
  // (Walsh coefficients akw_hi); kp counts the planes of the wider code
  int ksplit;
  float kc_hi[16], kt_hi[16], akw_hi[8];
  // byte key norms: code c > 0 decodes to 2^(kn_lo + (c - 1) kn_step)
  int knu8;
  float kn_lo, kn_step, kn_inv_step;
  int kp, vp;                          // 2^(bits-1) planes
  uint32_t xb1, xb2;                   // 0x3C003C00 and 0x40004000 (f16 pairs 1.0, 2.0), passed as data so
                                       // that an operand register stays one LOP3 with a register operand
  int sub_bytes;                       // bytes of one (page, head) sub-block
  int off_knorm, off_krnorm, off_kcodes, off_kx, off_ksigns, off_vnorm, off_vcodes;
  // KIVI arm: integer codes with float16 scale / zero (key per channel, value per token);
  // off_kcodes / off_vcodes hold the codes
  int kivi;
  int off_kscale, off_kzero, off_vscale, off_vzero;
};

// Byte key norm ([Design study] §Packed format, u8 log-norm): 0 for a zero
// vector, else 1 + round-half-up of (log2 n - lo) / step clamped to 0..254.
__device__ __forceinline__ uint8_t norm_u8_encode(float n, const KParams& P) {
  if (n < kZeroNorm) return 0;
  const float t = (log2f(n) - P.kn_lo) * P.kn_inv_step;
  const float k = fminf(fmaxf(floorf(t + 0.5f), 0.f), 254.f);
  return (uint8_t)(1 + (int)k);
}

__device__ __forceinline__ float norm_u8_decode(unsigned c, const KParams& P) {
  return c == 0 ? 0.f : exp2f(P.kn_lo + (float)(c - 1) * P.kn_step);
}

// Cache descriptor as seen by the kernels.
struct KCache {
  unsigned char* pool;
  long long n_pages;
  const int32_t* block_table;
  int max_pages;
  int32_t* seq_len;
  int32_t* n_compressed;
  __half* win_k;
  __half* win_v;
  int batch;
  int ring;                            // window + 16 (0 without window)
  // prefill attention: row b of seq_len / n_compressed is a virtual sequence (one query of a
  // chunk with its causal length) reading block-table row and window ring parent[b]; NULL = b
  const int32_t* parent;
};

__device__ __forceinline__ float load_elem(const void* p, int dtype, long long i) {
  if (dtype == TQ_F32) return __ldg(reinterpret_cast<const float*>(p) + i);
  if (dtype == TQ_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
  return __half2float(reinterpret_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Code index of z: #{i : z >= t_i} over the 2^bits - 1 boundaries.
__device__ __forceinline__ int bucketize(float z, const float* t, int bits) {
  const int nb = (1 << bits) - 1;
  int idx = 0;
#pragma unroll
  for (int i = 0; i < 15; ++i) idx += (i < nb && z >= t[i]) ? 1 : 0;
  return idx;
}

// Sign-magnitude plane bit p of code idx.
__device__ __forceinline__ unsigned plane_bit(int idx, int bits, int p) {
  const int half = 1 << (bits - 1);
  const bool pos = idx >= half;
  if (p == 0) return pos ? 1u : 0u;
  const int m = pos ? idx - half : half - 1 - idx;
  return (unsigned)((m >> (p - 1)) & 1);
}

// Centroid of a code given its sign bit and magnitude m.
__device__ __forceinline__ float centroid_sm(const float* c, int bits, unsigned pos, int m) {
  const int half = 1 << (bits - 1);
  return pos ? c[half + m] : c[half - 1 - m];
}

}  // namespace tq
