// Decode attention over the compressed paged cache (sm_103a).
//
// [Design study] §Transform placement: the query is moved into the rotated
// key basis once, scores are computed against the packed key codes, value
// pages are streamed after the softmax; §CPU and WASM kernel design: FP32
// score and output accumulators, value accumulation in the rotated value
// basis with ONE inverse transform per head.  [Reconstruction] §6: score
//   l = scale * n * ( <q', C[idx]> / sqrt(d) + sqrt(pi/2)/d * gamma * <q'', 2s - 1> ),
//   q' = Pi q, q'' = S q'.
//
// Three launches per call:
//   decode_prologue_kernel  grid (batch, Hkv):  q' and q'' for the G query
//                           heads of each kv head (tile product / FWHT).
//   decode_main_kernel      grid (splits + 1, Hkv, batch): split-K over the
//                           page list with an online softmax per split; the
//                           last split scans the float16 window in the
//                           unrotated basis.  Writes (m, l, acc[d]) partials.
//   decode_combine_kernel   grid (batch, Hkv): merges the partials in a fixed
//                           order (deterministic), applies Pi_v^T once to the
//                           rotated accumulator, adds the window part.
#include <math.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_launch.h"
#include "tq_tile.cuh"

namespace tq {

__device__ unsigned int g_decode_err = 0;

constexpr int kDecThreads = 256;
constexpr int kMaxSubBytes = 16 * (8 + 5 * 32) + 16 * (4 + 4 * 32);  // d = 256, 4+1 key bits, 4 value bits

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout decode_ws_layout(const KParams& P, int batch, int max_ctx, int n_splits, int num_sms) {
  WsLayout L{};
  const int max_pages = std::max(1, (max_ctx + kPage - 1) / kPage);
  int S = n_splits;
  if (S <= 0) {
    const int units = std::max(1, batch * P.hkv);
    S = (4 * num_sms + units - 1) / units;
    S = std::max(1, std::min(S, (max_pages + 3) / 4));
  }
  S = std::min(S, max_pages);
  const int pps = (max_pages + S - 1) / S;
  S = (max_pages + pps - 1) / pps;
  L.n_comp_splits = S;
  L.pages_per_split = pps;
  const size_t heads = (size_t)batch * P.hq;
  const int st = S + 1;
  size_t o = 0;
  L.qrot = o; o = align256(o + heads * P.d * sizeof(float));
  L.qsk = o;  o = align256(o + heads * P.d * sizeof(float));
  L.ml = o;   o = align256(o + heads * st * 2 * sizeof(float));
  L.acc = o;  o = align256(o + heads * st * (size_t)P.d * sizeof(float));
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ prologue

template <int D>
__global__ void __launch_bounds__(D) decode_prologue_kernel(const __grid_constant__ KParams P, const void* q,
                                                            int dtype, float* qrot, float* qsk) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<D>& s = *reinterpret_cast<TileSmem<D>*>(smem_raw);
  const int b = blockIdx.x, g = blockIdx.y, j = threadIdx.x;
  const int G = P.G;
  const size_t base = ((size_t)b * P.hq + (size_t)g * G) * D;
  for (int i = 0; i < G; ++i) s.x[i][j] = load_elem(q, dtype, (long long)(base + (size_t)i * D + j));
  if (j < G) s.inv[j] = P.kind == TQ_FWHT ? rsqrtf((float)D) : 1.0f;
  __syncthreads();
  rotate_tile<D>(s, G, P.kind, P.k_rot + (size_t)g * (P.kind == TQ_FWHT ? D : D * D));
  for (int i = 0; i < G; ++i) qrot[base + (size_t)i * D + j] = s.x[i][j];
  if (!P.kqjl) return;
  const float4* row = reinterpret_cast<const float4*>(P.qjl_s + (size_t)g * D * D + (size_t)j * D);
  float acc[TQ_MAX_GQA];
#pragma unroll
  for (int i = 0; i < TQ_MAX_GQA; ++i) acc[i] = 0.f;
  for (int i4 = 0; i4 < D / 4; ++i4) {
    const float4 p = __ldg(row + i4);
#pragma unroll
    for (int i = 0; i < TQ_MAX_GQA; ++i) {
      if (i < G) {
        const float4 xv = *reinterpret_cast<const float4*>(&s.x[i][i4 * 4]);
        acc[i] = fmaf(p.x, xv.x, fmaf(p.y, xv.y, fmaf(p.z, xv.z, fmaf(p.w, xv.w, acc[i]))));
      }
    }
  }
  for (int i = 0; i < G; ++i) qsk[base + (size_t)i * D + j] = acc[i];
}

// ------------------------------------------------------------------ main (split-K)

struct DecodeSmemCommon {
  float sc[kPage][TQ_MAX_GQA];
  float wt[kPage][TQ_MAX_GQA];
  float alpha[TQ_MAX_GQA];
  float mrun[TQ_MAX_GQA];
  float lrun[TQ_MAX_GQA];
  float ck[16], cv[16];
  float red[kDecThreads][TQ_MAX_GQA];
};

// Online-softmax update for one block of 16 scores (thread h < G).
template <int G>
__device__ __forceinline__ void softmax_block(DecodeSmemCommon& c, const float* vnorm, float wscale) {
  const int h = threadIdx.x;
  if (h < G) {
    float mx = -INFINITY;
#pragma unroll
    for (int t = 0; t < kPage; ++t) mx = fmaxf(mx, c.sc[t][h]);
    const float mold = c.mrun[h];
    const float mnew = fmaxf(mold, mx);
    if (mnew == -INFINITY) {
      c.alpha[h] = 1.f;
#pragma unroll
      for (int t = 0; t < kPage; ++t) c.wt[t][h] = 0.f;
    } else {
      const float a = expf(mold - mnew);
      float sum = 0.f;
#pragma unroll
      for (int t = 0; t < kPage; ++t) {
        const float e = expf(c.sc[t][h] - mnew);
        sum += e;
        c.wt[t][h] = e > 0.f ? e * (vnorm ? vnorm[t] * wscale : 1.0f) : 0.f;
      }
      c.alpha[h] = a;
      c.lrun[h] = c.lrun[h] * a + sum;
      c.mrun[h] = mnew;
    }
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads) decode_main_kernel(const __grid_constant__ KParams P,
                                                                   const __grid_constant__ KCache C, const void* q,
                                                                   int dtype, float scale, float* scores,
                                                                   unsigned char* ws, WsLayout L, int max_ctx) {
  constexpr int E = D / 32;
  constexpr int NGRP = kDecThreads / D;      // token groups in the value phase
  constexpr int TPG = kPage / NGRP;          // tokens per group
  extern __shared__ __align__(16) unsigned char dyn[];
  __shared__ DecodeSmemCommon c;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nsplit_tot = L.n_comp_splits + 1;
  const bool window_split = s == L.n_comp_splits;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float kappa = sqrtf(1.57079632679489662f) / (float)D;

  int T = C.seq_len[b];
  int nc = C.n_compressed[b];
  if (T < 0 || T > max_ctx || nc < 0 || nc > T) {
    if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
    T = min(max(T, 0), max_ctx);
    nc = min(max(nc, 0), T);
  }
  if (tid < 16) {
    c.ck[tid] = P.kc[tid];
    c.cv[tid] = P.vc[tid];
  }
  if (tid < G) {
    c.mrun[tid] = -INFINITY;
    c.lrun[tid] = 0.f;
  }
  float accv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) accv[h] = 0.f;
  const int cj = tid % D, grp = tid / D;
  const size_t head0 = (size_t)b * P.hq + (size_t)g * G;

  if (!window_split) {
    int np = (nc + kPage - 1) / kPage;
    if (np > C.max_pages) {
      if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
      np = C.max_pages;
    }
    const int p0 = s * L.pages_per_split;
    const int p1 = min(p0 + L.pages_per_split, np);
    const float* qrot = reinterpret_cast<const float*>(ws + L.qrot);
    const float* qsk = reinterpret_cast<const float*>(ws + L.qsk);
    float qa[G][E], qb[G][E];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        qa[h][e] = qrot[(head0 + h) * D + e * 32 + lane];
        qb[h][e] = P.kqjl ? qsk[(head0 + h) * D + e * 32 + lane] : 0.f;
      }
    unsigned char* pb = dyn;
    const int kbits = P.kb, vbits = P.vb;
    const int khalf = 1 << (kbits - 1), vhalf = 1 << (vbits - 1);
    __syncthreads();
    for (int p = p0; p < p1; ++p) {
      const long long pid = C.block_table[(size_t)b * C.max_pages + p];
      const bool pvalid = pid >= 0 && pid < C.n_pages;
      if (!pvalid && tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_PAGE_INDEX);
      if (pvalid) {
        const uint4* src = reinterpret_cast<const uint4*>(C.pool + ((size_t)pid * P.hkv + g) * (size_t)P.sub_bytes);
        uint4* dst = reinterpret_cast<uint4*>(pb);
        for (int i = tid; i < P.sub_bytes / 16; i += kDecThreads) dst[i] = __ldg(src + i);
      }
      __syncthreads();
      const float* knorm = reinterpret_cast<const float*>(pb + P.off_knorm);
      const float* krn = reinterpret_cast<const float*>(pb + P.off_krnorm);
      const uint32_t* kc = reinterpret_cast<const uint32_t*>(pb + P.off_kcodes);
      const uint32_t* ks = reinterpret_cast<const uint32_t*>(pb + P.off_ksigns);
      const float* vnorm = reinterpret_cast<const float*>(pb + P.off_vnorm);
      const uint16_t* vc = reinterpret_cast<const uint16_t*>(pb + P.off_vcodes);
      // scores: warp w handles tokens w and w + 8
      for (int t = warp; t < kPage; t += kDecThreads / 32) {
        const int tok = p * kPage + t;
        const bool live = pvalid && tok < nc;
        float am[G], aq[G];
#pragma unroll
        for (int h = 0; h < G; ++h) am[h] = aq[h] = 0.f;
        if (live) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const unsigned pos = (kc[(0 * kPage + t) * E + e] >> lane) & 1u;
            int m = 0;
            for (int pl = 1; pl < kbits; ++pl) m |= (int)((kc[(pl * kPage + t) * E + e] >> lane) & 1u) << (pl - 1);
            const float cval = pos ? c.ck[khalf + m] : c.ck[khalf - 1 - m];
#pragma unroll
            for (int h = 0; h < G; ++h) am[h] = fmaf(cval, qa[h][e], am[h]);
            if (P.kqjl) {
              const bool sg = (ks[t * E + e] >> lane) & 1u;
#pragma unroll
              for (int h = 0; h < G; ++h) aq[h] += sg ? qb[h][e] : -qb[h][e];
            }
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          am[h] = warp_sum_f(am[h]);
          aq[h] = warp_sum_f(aq[h]);
        }
        if (lane == 0) {
          const float n = live ? knorm[t] : 0.f;
          const float gm = (live && P.kqjl) ? krn[t] : 0.f;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float l = live ? scale * n * (am[h] * inv_sqrt_d + kappa * gm * aq[h]) : -INFINITY;
            c.sc[t][h] = l;
            if (scores && live) scores[(head0 + h) * (size_t)max_ctx + tok] = l;
          }
        }
      }
      __syncthreads();
      softmax_block<G>(c, vnorm, inv_sqrt_d);
      __syncthreads();
      // values (rotated basis): thread (cj, grp) over its token group
      {
        float a[G];
#pragma unroll
        for (int h = 0; h < G; ++h) a[h] = accv[h] * c.alpha[h];
        unsigned w[TQ_MAX_BITS];
#pragma unroll
        for (int pl = 0; pl < TQ_MAX_BITS; ++pl) w[pl] = pl < vbits ? vc[pl * D + cj] : 0u;
#pragma unroll
        for (int tt = 0; tt < TPG; ++tt) {
          const int t = grp * TPG + tt;
          const unsigned pos = (w[0] >> t) & 1u;
          int m = 0;
#pragma unroll
          for (int pl = 1; pl < TQ_MAX_BITS; ++pl) m |= (int)((w[pl] >> t) & 1u) << (pl - 1);
          const float cval = pos ? c.cv[vhalf + (m & (vhalf - 1))] : c.cv[vhalf - 1 - (m & (vhalf - 1))];
#pragma unroll
          for (int h = 0; h < G; ++h) a[h] = fmaf(c.wt[t][h], cval, a[h]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) accv[h] = a[h];
      }
      __syncthreads();
    }
  } else {
    // window split: tokens nc .. T-1 from the float16 ring, unrotated basis
    float* qs = reinterpret_cast<float*>(dyn);                 // [G][D]
    float* kw = qs + G * D;                                     // [16][D]
    float* vw = kw + kPage * D;                                 // [16][D]
    for (int i = tid; i < G * D; i += kDecThreads) qs[i] = load_elem(q, dtype, (long long)(head0 * D + i));
    int nw = T - nc;
    if (nw > 0 && (C.ring == 0 || nw > C.ring)) {
      if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
      nw = C.ring == 0 ? 0 : min(nw, C.ring);
    }
    __syncthreads();
    for (int c0 = 0; c0 < nw; c0 += kPage) {
      for (int i = tid; i < kPage * D; i += kDecThreads) {
        const int t = i / D, jj = i % D;
        float kv = 0.f, vv = 0.f;
        if (c0 + t < nw && C.win_k) {
          const size_t slot = (size_t)((nc + c0 + t) % C.ring);
          const size_t off = (((size_t)b * P.hkv + g) * C.ring + slot) * D + jj;
          kv = __half2float(C.win_k[off]);
          vv = __half2float(C.win_v[off]);
        }
        kw[i] = kv;
        vw[i] = vv;
      }
      __syncthreads();
      for (int t = warp; t < kPage; t += kDecThreads / 32) {
        const bool live = c0 + t < nw;
        float a[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) acc = fmaf(qs[h * D + e * 32 + lane], kw[t * D + e * 32 + lane], acc);
          a[h] = warp_sum_f(acc);
        }
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float l = live ? scale * a[h] : -INFINITY;
            c.sc[t][h] = l;
            if (scores && live) scores[(head0 + h) * (size_t)max_ctx + nc + c0 + t] = l;
          }
        }
      }
      __syncthreads();
      softmax_block<G>(c, nullptr, 1.f);
      __syncthreads();
      {
        float a[G];
#pragma unroll
        for (int h = 0; h < G; ++h) a[h] = accv[h] * c.alpha[h];
#pragma unroll
        for (int tt = 0; tt < TPG; ++tt) {
          const int t = grp * TPG + tt;
          const float vv = vw[t * D + cj];
#pragma unroll
          for (int h = 0; h < G; ++h) a[h] = fmaf(c.wt[t][h], vv, a[h]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) accv[h] = a[h];
      }
      __syncthreads();
    }
  }
  // partials: reduce token groups, then store (m, l, acc)
  __syncthreads();
#pragma unroll
  for (int h = 0; h < G; ++h) c.red[tid][h] = accv[h];
  __syncthreads();
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  if (tid < D) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v = 0.f;
#pragma unroll
      for (int gr = 0; gr < NGRP; ++gr) v += c.red[gr * D + tid][h];
      acc[((head0 + h) * nsplit_tot + s) * D + tid] = v;
    }
  }
  if (tid < G) {
    ml[((head0 + tid) * nsplit_tot + s) * 2 + 0] = c.mrun[tid];
    ml[((head0 + tid) * nsplit_tot + s) * 2 + 1] = c.lrun[tid];
  }
}

// ------------------------------------------------------------------ combine

template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const __grid_constant__ KParams P,
                                                           const unsigned char* ws, WsLayout L, float* out,
                                                           float* lse) {
  constexpr int E = D / 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<D>& s = *reinterpret_cast<TileSmem<D>*>(smem_raw);
  __shared__ float Ms[TQ_MAX_GQA], Ls[TQ_MAX_GQA];
  const int b = blockIdx.x, g = blockIdx.y, j = threadIdx.x, lane = j & 31, warp = j >> 5;
  const int G = P.G;
  const int st = L.n_comp_splits + 1;
  const size_t head0 = (size_t)b * P.hq + (size_t)g * G;
  const float* ml = reinterpret_cast<const float*>(ws + L.ml);
  const float* acc = reinterpret_cast<const float*>(ws + L.acc);
  for (int i = 0; i < G; ++i) {
    const float* mli = ml + (head0 + i) * st * 2;
    float M = -INFINITY;
    for (int k = 0; k < st; ++k) M = fmaxf(M, mli[2 * k]);
    float Lsum = 0.f, rot = 0.f, win = 0.f;
    if (M != -INFINITY) {
      for (int k = 0; k < st; ++k) {
        const float m = mli[2 * k];
        if (m == -INFINITY) continue;
        const float f = expf(m - M);
        Lsum += mli[2 * k + 1] * f;
        const float a = acc[((head0 + i) * st + k) * D + j] * f;
        if (k < st - 1) rot += a;
        else win += a;
      }
    }
    s.x[i][j] = rot;
    s.r[i][j] = win;
    if (j == 0) {
      Ms[i] = M;
      Ls[i] = Lsum;
    }
  }
  __syncthreads();
  // inverse value rotation Pi_v^T, once per head
  const float* vrot = P.v_rot + (size_t)g * (P.kind == TQ_FWHT ? D : D * D);
  if (P.kind == TQ_FWHT) {
    // Pi^T y = sigma * (H y) / sqrt(d)
    for (int v = warp; v < G; v += D / 32) {
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = s.x[v][e * 32 + lane];
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
      const float sc = rsqrtf((float)D);
#pragma unroll
      for (int e = 0; e < E; ++e) s.x[v][e * 32 + lane] = a[e] * sc * __ldg(vrot + e * 32 + lane);
    }
    __syncthreads();
  } else {
    float o[TQ_MAX_GQA];
#pragma unroll
    for (int i = 0; i < TQ_MAX_GQA; ++i) o[i] = 0.f;
    for (int jj = 0; jj < D; ++jj) {
      const float pv = __ldg(vrot + (size_t)jj * D + j);  // column j of Pi_v
#pragma unroll
      for (int i = 0; i < TQ_MAX_GQA; ++i)
        if (i < G) o[i] = fmaf(pv, s.x[i][jj], o[i]);
    }
    __syncthreads();
    for (int i = 0; i < G; ++i) s.x[i][j] = o[i];
    __syncthreads();
  }
  for (int i = 0; i < G; ++i) {
    const float M = Ms[i], Lsum = Ls[i];
    const bool empty = M == -INFINITY || Lsum <= 0.f;
    out[(head0 + i) * D + j] = empty ? 0.f : (s.x[i][j] + s.r[i][j]) / Lsum;
    if (lse && j == 0) lse[head0 + i] = empty ? -INFINITY : M + logf(Lsum);
  }
}

// ------------------------------------------------------------------ launcher

template <int D, int G>
static cudaError_t launch_main(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                               float* scores, unsigned char* ws, const WsLayout& L, int max_ctx, int batch,
                               cudaStream_t st) {
  const size_t dyn = std::max<size_t>((size_t)kMaxSubBytes, (size_t)(G * D + 2 * kPage * D) * sizeof(float));
  cudaError_t e = cudaFuncSetAttribute(decode_main_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  dim3 grid(L.n_comp_splits + 1, P.hkv, batch);
  decode_main_kernel<D, G><<<grid, kDecThreads, dyn, st>>>(P, C, q, dtype, scale, scores, ws, L, max_ctx);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_main_g(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                                 float* scores, unsigned char* ws, const WsLayout& L, int max_ctx, int batch,
                                 cudaStream_t st) {
  switch (P.G) {
    case 1: return launch_main<D, 1>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
    case 2: return launch_main<D, 2>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
    case 3: return launch_main<D, 3>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
    case 4: return launch_main<D, 4>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
    case 5: return launch_main<D, 5>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
    case 6: return launch_main<D, 6>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
    case 7: return launch_main<D, 7>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
    default: return launch_main<D, 8>(P, C, q, dtype, scale, scores, ws, L, max_ctx, batch, st);
  }
}

template <int D>
static cudaError_t launch_decode_d(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                                   float* out, float* lse, float* scores, void* ws, const WsLayout& L, int max_ctx,
                                   cudaStream_t st) {
  unsigned char* w = reinterpret_cast<unsigned char*>(ws);
  const size_t tsm = sizeof(TileSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(decode_prologue_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsm);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_combine_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsm);
  if (e != cudaSuccess) return e;
  dim3 g2(C.batch, P.hkv);
  decode_prologue_kernel<D><<<g2, D, tsm, st>>>(P, q, dtype, reinterpret_cast<float*>(w + L.qrot),
                                                reinterpret_cast<float*>(w + L.qsk));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_main_g<D>(P, C, q, dtype, scale, scores, w, L, max_ctx, C.batch, st)) != cudaSuccess) return e;
  decode_combine_kernel<D><<<g2, D, tsm, st>>>(P, w, L, out, lse);
  return cudaGetLastError();
}

cudaError_t launch_decode(const KParams& P, const KCache& C, const void* q, int dtype, float scale, float* out,
                          float* lse, float* scores, void* ws, const WsLayout& L, int max_ctx, cudaStream_t st) {
  if (P.d == 128) return launch_decode_d<128>(P, C, q, dtype, scale, out, lse, scores, ws, L, max_ctx, st);
  return launch_decode_d<256>(P, C, q, dtype, scale, out, lse, scores, ws, L, max_ctx, st);
}

cudaError_t read_clear_decode_error(unsigned* bits) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_decode_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(unsigned));
}

}  // namespace tq
