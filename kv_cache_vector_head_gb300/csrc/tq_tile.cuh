// Tile routines shared by the quantize, append and decode kernels: a tile is
// up to 16 vectors of one kv head held in shared memory, blockDim == d.
#pragma once

#include "tq_device.cuh"

namespace tq {

template <int D>
struct TileSmem {
  float x[kTile][D + 4];      // input, then z
  float r[kTile][D + 4];      // dense rotation output / scaled residual
  float inv[kTile];
  float norm[kTile];
  float gam[kTile];
  int zero[kTile];
  uint32_t codes[kTile][TQ_MAX_BITS][D / 32];
  uint32_t signs[kTile][D / 32];
  uint32_t vmask[TQ_MAX_BITS][D];  // coordinate-major value bits per slot
  float cb[16], tb[16];
  float cb_hi[16], tb_hi[16];      // mixed-channel keys: the book of coordinates < d/2
};

// In-register Walsh-Hadamard transform of one d-vector held by a warp
// (coordinate e * 32 + lane in a[e]); unnormalised, Sylvester order.
template <int E>
__device__ __forceinline__ void warp_wht(float (&a)[E], int lane) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float o = __shfl_xor_sync(0xffffffffu, a[e], h);
      a[e] = (lane & h) ? (o - a[e]) : (a[e] + o);
    }
  }
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if ((e & h) == 0) {
        const float lo = a[e], hi = a[e + h];
        a[e] = lo + hi;
        a[e + h] = lo - hi;
      }
    }
  }
}

// out[v][j] = inv[v] * (R x_v)_j, R = Pi (dense) or H diag(sigma) (FWHT).
// In place in s.x (the dense product goes through registers).
template <int D, int MAXV = kTile>
__device__ void rotate_tile(TileSmem<D>& s, int nv, int kind, const float* rot) {
  constexpr int E = D / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (kind == TQ_FWHT) {
    for (int v = warp; v < nv; v += D / 32) {
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = s.x[v][e * 32 + lane] * __ldg(rot + e * 32 + lane);
      warp_wht<E>(a, lane);
      const float sc = s.inv[v];
#pragma unroll
      for (int e = 0; e < E; ++e) s.x[v][e * 32 + lane] = a[e] * sc;
    }
    __syncthreads();
  } else {
    const int j = tid;
    float acc[MAXV];
#pragma unroll
    for (int v = 0; v < MAXV; ++v) acc[v] = 0.f;
    const float4* row = reinterpret_cast<const float4*>(rot + (size_t)j * D);
#pragma unroll 8
    for (int i4 = 0; i4 < D / 4; ++i4) {
      const float4 p = __ldg(row + i4);
#pragma unroll
      for (int v = 0; v < MAXV; ++v) {
        if (v < nv) {
          const float4 xv = *reinterpret_cast<const float4*>(&s.x[v][i4 * 4]);
          acc[v] = fmaf(p.x, xv.x, acc[v]);
          acc[v] = fmaf(p.y, xv.y, acc[v]);
          acc[v] = fmaf(p.z, xv.z, acc[v]);
          acc[v] = fmaf(p.w, xv.w, acc[v]);
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int v = 0; v < MAXV; ++v)
      if (v < nv) s.x[v][j] = acc[v] * s.inv[v];
    __syncthreads();
  }
}

}  // namespace tq
