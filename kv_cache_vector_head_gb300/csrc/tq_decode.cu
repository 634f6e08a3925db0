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
// The two contractions of a decode step are dense products over the G query
// heads of a KV head:  scores[h, t] = sum_j Q[h, j] K_hat[t, j] and
// acc[h, j] = sum_t w[h, t] V_hat[t, j].  They run on the tensor cores
// (mma.m16n8k16, f16 operands, f32 accumulation) with operands that are
// EXACT in f16:
//   * a b-bit code with sign s and magnitude bits m has centroid
//     s * sum_S a_S prod_{i in S} (1 - 2 m_i) (Walsh expansion over the
//     magnitude bits), so the token side is a sum of +-1 "planes" P_S whose
//     sign bit is s ^ parity(m & S) -- built from the packed words with one
//     shift and one LOP3 per pair of coordinates, no lookup;
//   * the query side a_S q' (and q'') and the softmax weights are split into
//     f16 hi + lo limbs that occupy rows h and h + 8 of the 16-row tile
//     (G <= 8 heads), so the second limb costs no extra instruction;
//   * values with b >= 3 bits use f16 hi / lo limbs of the centroid itself
//     (two planes) read from a 16-entry table, instead of 2^(b-1) planes.
// Every product is exact and accumulation is f32, so the scores carry
// ~2^-22 relative query rounding instead of f16's 2^-11.
//
// Launches per call:
//   decode_prologue_kernel  grid (Hq, batch): q' = Pi q, q'' = S q' and this
//                           head's rows of the query fragments (mma order).
//   decode_window_kernel    grid (Hkv, batch): the float16 window, unrotated
//                           basis, CUDA cores (at most W + 15 tokens).
//   decode_mma_kernel       grid (splits, Hkv, batch): split-K over the page
//                           list.  Pages stream into shared memory with 1-D
//                           TMA bulk copies (cp.async.bulk + mbarrier, three
//                           stages of 4 pages); warp w scores page w of each
//                           4-page chunk, then all warps accumulate values for
//                           their quarter of the coordinates.
//   decode_combine_kernel   grid (Hq, batch): merges the partials in a fixed
//                           order, applies Pi_v^T once, adds the window part.
#include <math.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_launch.h"
#include "tq_tile.cuh"

namespace tq {

__device__ unsigned int g_decode_err = 0;

constexpr int kMmaThreads = 128;
constexpr int kChunkPages = 4;
constexpr int kStages = 3;
constexpr int kWinThreads = 128;
constexpr unsigned kWaitLimit = 1u << 24;  // bounded mbarrier polling

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int key_frag_planes(const KParams& P) { return P.kp + (P.kqjl ? 1 : 0); }

WsLayout decode_ws_layout(const KParams& P, int batch, int max_ctx, int n_splits, int num_sms) {
  WsLayout L{};
  const int max_pages = std::max(1, (max_ctx + kPage - 1) / kPage);
  int S = n_splits;
  if (S <= 0) {
    const int units = std::max(1, batch * P.hkv);
    S = (3 * num_sms + units - 1) / units;
    S = std::max(1, std::min(S, (max_pages + 7) / 8));
  }
  S = std::min(S, max_pages);
  const int pps = (max_pages + S - 1) / S;
  S = (max_pages + pps - 1) / pps;
  L.n_comp_splits = S;
  L.pages_per_split = pps;
  const size_t heads = (size_t)batch * P.hq;
  const int st = S + 1;
  L.afrag_bytes_per_head = (size_t)key_frag_planes(P) * (P.d / 16) * 32 * 16;
  size_t o = 0;
  L.afrag = o; o = align256(o + (size_t)batch * P.hkv * L.afrag_bytes_per_head);
  L.ml = o;    o = align256(o + heads * st * 2 * sizeof(float));
  L.acc = o;   o = align256(o + heads * st * (size_t)P.d * sizeof(float));
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint4& a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// f16 pair (+-1, +-1) from bits i and i + 16 of nw = ~plane_word (bit set -> -1).
__device__ __forceinline__ uint32_t pm1_pair(uint32_t nw, int i) {
  return ((nw << (15 - i)) & 0x80008000u) | 0x3C003C00u;
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

__device__ __forceinline__ void split_f16(float v, __half& hi, __half& lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false if the phase did not complete within kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (unsigned i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// In-register Walsh-Hadamard transform of one d-vector held by a warp
// (coordinate e * 32 + lane in a[e]); unnormalised, Sylvester order.
template <int E>
__device__ __forceinline__ void warp_fwht(float (&a)[E], int lane) {
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

// ------------------------------------------------------------------ prologue

// One CTA per (query head h, sequence): q' = Pi_g q and q'' = S_g q' (g the
// kv head of h), then this head's rows of the query operand of the score
// products, in mma.m16n8k16 A-fragment order:
//   frag[plane][kk][lane] = 4 x f16x2, rows h_local (hi limb) and h_local + 8
//   (lo limb), k-pair (2t, 2t+1) <-> bits (i0, i0+16) and (2t+8, 2t+9) <->
//   (i0+1, i0+17) of plane word w = t * (d/128) + kk / 8, i0 = 2 (kk mod 8),
//   t = lane mod 4.  Rows of absent heads (h_local >= G) are zero.
template <int D>
__global__ void __launch_bounds__(D) decode_prologue_kernel(const __grid_constant__ KParams P, const void* q,
                                                            int dtype, unsigned char* ws, WsLayout L) {
  constexpr int KS = D / 16, WPL = D / 128, E = D / 32;
  __shared__ float qr[D], qs[D];
  const int hq = blockIdx.x, b = blockIdx.y, j = threadIdx.x, lane = j & 31, warp = j >> 5;
  const int G = P.G, g = hq / G, hl = hq % G;
  const size_t qoff = ((size_t)b * P.hq + hq) * D;
  if (P.kind == TQ_FWHT) {
    if (warp == 0) {
      const float* sg = P.k_rot + (size_t)g * D;
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e)
        a[e] = load_elem(q, dtype, (long long)(qoff + e * 32 + lane)) * __ldg(sg + e * 32 + lane);
      warp_fwht<E>(a, lane);
      const float sc = rsqrtf((float)D);
#pragma unroll
      for (int e = 0; e < E; ++e) qr[e * 32 + lane] = a[e] * sc;
    }
  } else {
    qs[j] = load_elem(q, dtype, (long long)(qoff + j));
    __syncthreads();
    const float4* row = reinterpret_cast<const float4*>(P.k_rot + (size_t)g * D * D + (size_t)j * D);
    float acc = 0.f;
#pragma unroll 8
    for (int i4 = 0; i4 < D / 4; ++i4) {
      const float4 p = __ldg(row + i4);
      acc = fmaf(p.x, qs[4 * i4], fmaf(p.y, qs[4 * i4 + 1], fmaf(p.z, qs[4 * i4 + 2], fmaf(p.w, qs[4 * i4 + 3], acc))));
    }
    qr[j] = acc;
  }
  __syncthreads();
  if (P.kqjl) {
    const float4* row = reinterpret_cast<const float4*>(P.qjl_s + (size_t)g * D * D + (size_t)j * D);
    float acc = 0.f;
#pragma unroll 8
    for (int i4 = 0; i4 < D / 4; ++i4) {
      const float4 p = __ldg(row + i4);
      acc = fmaf(p.x, qr[4 * i4], fmaf(p.y, qr[4 * i4 + 1], fmaf(p.z, qr[4 * i4 + 2], fmaf(p.w, qr[4 * i4 + 3], acc))));
    }
    __syncthreads();
    qs[j] = acc;
  }
  __syncthreads();
  const int nplanes = P.kp + (P.kqjl ? 1 : 0);
  uint32_t* frag = reinterpret_cast<uint32_t*>(ws + L.afrag + ((size_t)b * P.hkv + g) * L.afrag_bytes_per_head);
  // this head's entries: lanes with lane / 4 == hl; head 0 also zeroes the rows of absent heads
  const int nrow = (hl == 0) ? (8 - G + 1) : 1;
  const int total = nplanes * KS * 4 * 4 * nrow;
  for (int idx = j; idx < total; idx += D) {
    const int r = idx & 3, t4 = (idx >> 2) & 3, rest = idx >> 4;
    const int rowsel = rest % nrow, kk = (rest / nrow) % KS, pl = (rest / nrow) / KS;
    const int g8 = rowsel == 0 ? hl : (G - 1 + rowsel);
    const int lanei = g8 * 4 + t4;
    uint32_t val = 0;
    if (rowsel == 0) {
      const int w = t4 * WPL + kk / 8, i0 = 2 * (kk % 8) + ((r >= 2) ? 1 : 0);
      const int ca = 32 * w + i0, cb = ca + 16;
      float va, vb;
      if (pl < P.kp) {
        va = P.akw[pl] * qr[ca];
        vb = P.akw[pl] * qr[cb];
      } else {
        va = qs[ca];
        vb = qs[cb];
      }
      __half ha, la, hb, lb;
      split_f16(va, ha, la);
      split_f16(vb, hb, lb);
      val = (r & 1) ? pack_h2(la, lb) : pack_h2(ha, hb);
    }
    frag[((pl * KS + kk) * 32 + lanei) * 4 + r] = val;
  }
}

// ------------------------------------------------------------------ window (CUDA cores)

// One CTA per (kv head, sequence): scores of every window token for the G
// heads (one warp per token), one softmax per head over the window, then the
// weighted sum of the float16 values (thread per coordinate).
template <int D>
__global__ void __launch_bounds__(kWinThreads) decode_window_kernel(const __grid_constant__ KParams P,
                                                                    const __grid_constant__ KCache C,
                                                                    const void* q, int dtype, float scale,
                                                                    float* scores, unsigned char* ws, WsLayout L,
                                                                    int max_ctx) {
  constexpr int E = D / 32, CPT = D / kWinThreads;
  extern __shared__ __align__(16) float wsc[];  // [ring][TQ_MAX_GQA] scores, then weights
  __shared__ float qs[TQ_MAX_GQA][D];
  __shared__ float mx_s[TQ_MAX_GQA], sum_s[TQ_MAX_GQA];
  const int g = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = P.G;
  const int st = L.n_comp_splits + 1;
  const size_t head0 = (size_t)b * P.hq + (size_t)g * G;
  int T = C.seq_len[b], nc = C.n_compressed[b];
  if (T < 0 || T > max_ctx || nc < 0 || nc > T) {
    if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
    T = min(max(T, 0), max_ctx);
    nc = min(max(nc, 0), T);
  }
  int nw = T - nc;
  if (nw > 0 && (C.ring == 0 || nw > C.ring)) {
    if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
    nw = C.ring == 0 ? 0 : min(nw, C.ring);
  }
  for (int i = tid; i < G * D; i += kWinThreads) qs[i / D][i % D] = load_elem(q, dtype, (long long)(head0 * D + i));
  __syncthreads();
  const size_t ring0 = ((size_t)b * P.hkv + g) * (size_t)C.ring;
  for (int t = warp; t < nw; t += kWinThreads / 32) {
    const __half* kr = C.win_k + (ring0 + (size_t)((nc + t) % C.ring)) * D;
    float kv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) kv[e] = __half2float(kr[e * 32 + lane]);
    for (int h = 0; h < G; ++h) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) a = fmaf(qs[h][e * 32 + lane], kv[e], a);
      a = warp_sum_f(a);
      if (lane == 0) {
        wsc[t * TQ_MAX_GQA + h] = scale * a;
        if (scores) scores[(head0 + h) * (size_t)max_ctx + nc + t] = scale * a;
      }
    }
  }
  __syncthreads();
  // per-head max and sum: warp h handles head h, lanes stride the tokens
  for (int h = warp; h < G; h += kWinThreads / 32) {
    float m = -INFINITY;
    for (int t = lane; t < nw; t += 32) m = fmaxf(m, wsc[t * TQ_MAX_GQA + h]);
    m = warp_max_f(m);
    float sm = 0.f;
    for (int t = lane; t < nw; t += 32) {
      const float e = expf(wsc[t * TQ_MAX_GQA + h] - m);
      wsc[t * TQ_MAX_GQA + h] = e;
      sm += e;
    }
    sm = warp_sum_f(sm);
    if (lane == 0) {
      mx_s[h] = m;
      sum_s[h] = sm;
    }
  }
  __syncthreads();
  float acc[TQ_MAX_GQA][CPT];
#pragma unroll
  for (int h = 0; h < TQ_MAX_GQA; ++h)
#pragma unroll
    for (int c = 0; c < CPT; ++c) acc[h][c] = 0.f;
  for (int t = 0; t < nw; ++t) {
    const __half* vr = C.win_v + (ring0 + (size_t)((nc + t) % C.ring)) * D;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const float vv = __half2float(vr[tid + c * kWinThreads]);
#pragma unroll
      for (int h = 0; h < TQ_MAX_GQA; ++h)
        if (h < G) acc[h][c] = fmaf(wsc[t * TQ_MAX_GQA + h], vv, acc[h][c]);
    }
  }
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  float* accw = reinterpret_cast<float*>(ws + L.acc);
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < CPT; ++c) accw[((head0 + h) * st + (st - 1)) * D + tid + c * kWinThreads] = acc[h][c];
  if (tid < G) {
    ml[((head0 + tid) * st + (st - 1)) * 2 + 0] = nw > 0 ? mx_s[tid] : -INFINITY;
    ml[((head0 + tid) * st + (st - 1)) * 2 + 1] = nw > 0 ? sum_s[tid] : 0.f;
  }
}

// ------------------------------------------------------------------ compressed pages (tensor cores)

struct MmaShared {
  uint64_t full[kStages];
  int pvalid[kStages][kChunkPages];
  float wsm[kChunkPages * kPage][TQ_MAX_GQA];  // weights of the chunk's 64 tokens
  float redm[kChunkPages][TQ_MAX_GQA];
  float reds[kChunkPages][TQ_MAX_GQA];
  float mrun[TQ_MAX_GQA], lrun[TQ_MAX_GQA], alpha[TQ_MAX_GQA];
  uint32_t vlut[16];  // values with b >= 3: raw sign-magnitude bits -> (hi, lo) f16 of the centroid
  int abort;
};

template <int D, bool VLUT>
__global__ void __launch_bounds__(kMmaThreads) decode_mma_kernel(const __grid_constant__ KParams P,
                                                                 const __grid_constant__ KCache C, float scale,
                                                                 float* scores, unsigned char* ws, WsLayout L,
                                                                 int max_ctx) {
  constexpr int E = D / 32, WPL = D / 128, KS = D / 16;
  constexpr int CPW = D / 4;         // value coordinates per warp
  constexpr int CB = CPW / 8;        // n-tiles per value plane per warp
  constexpr int VPL = 2;             // value planes held (Walsh b <= 2, or LUT hi / lo)
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ MmaShared sh;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, t4 = lane & 3;
  const int G = P.G;
  const int st = L.n_comp_splits + 1;
  const size_t head0 = (size_t)b * P.hq + (size_t)g * G;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float kappa = sqrtf(1.57079632679489662f) / (float)D;
  const int sub = P.sub_bytes;

  // shared memory: query fragments, then the page stages
  uint4* afr = reinterpret_cast<uint4*>(dyn);                        // [nkp][KS][32]
  unsigned char* stage0 = dyn + L.afrag_bytes_per_head;              // [kStages][4][sub]

  int T = C.seq_len[b], nc = C.n_compressed[b];
  if (T < 0 || T > max_ctx || nc < 0 || nc > T) {
    if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
    T = min(max(T, 0), max_ctx);
    nc = min(max(nc, 0), T);
  }
  int np = (nc + kPage - 1) / kPage;
  if (np > C.max_pages) {
    if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
    np = C.max_pages;
  }
  const int p0 = s * L.pages_per_split;
  const int p1 = min(p0 + L.pages_per_split, np);
  const int nchunks = p1 > p0 ? (p1 - p0 + kChunkPages - 1) / kChunkPages : 0;

  {
    const uint4* src = reinterpret_cast<const uint4*>(ws + L.afrag + ((size_t)b * P.hkv + g) * L.afrag_bytes_per_head);
    for (int i = tid; i < (int)(L.afrag_bytes_per_head / 16); i += kMmaThreads) afr[i] = src[i];
  }
  if (tid < TQ_MAX_GQA) {
    sh.mrun[tid] = -INFINITY;
    sh.lrun[tid] = 0.f;
    sh.alpha[tid] = 1.f;
  }
  for (int i = tid; i < kChunkPages * kPage * TQ_MAX_GQA; i += kMmaThreads) (&sh.wsm[0][0])[i] = 0.f;
  if (VLUT && tid < 16) {
    const int vb = P.vb, half = 1 << (vb - 1);
    uint32_t e = 0;
    if (tid < (1 << vb)) {
      const int sgn = tid & 1, m = tid >> 1;
      const float c = sgn ? P.vc[half + m] : P.vc[half - 1 - m];
      __half hi, lo;
      split_f16(c, hi, lo);
      e = pack_h2(hi, lo);
    }
    sh.vlut[tid] = e;
  }
  if (tid == 0) {
    sh.abort = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(&sh.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // producer (thread 0): chunk k = pages p0 + 4k .. into stage k % kStages
  auto issue = [&](int k) {
    const int stg = k % kStages;
    unsigned char* dst = stage0 + (size_t)stg * kChunkPages * sub;
    uint32_t bytes = 0;
    long long pids[kChunkPages];
#pragma unroll
    for (int i = 0; i < kChunkPages; ++i) {
      const int p = p0 + k * kChunkPages + i;
      long long pid = -1;
      if (p < p1) {
        pid = C.block_table[(size_t)b * C.max_pages + p];
        if (pid < 0 || pid >= C.n_pages) {
          atomicOr(&g_decode_err, TQ_DEVERR_PAGE_INDEX);
          pid = -1;
        }
      }
      pids[i] = pid;
      sh.pvalid[stg][i] = pid >= 0;
      if (pid >= 0) bytes += (uint32_t)sub;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(&sh.full[stg], bytes);
#pragma unroll
    for (int i = 0; i < kChunkPages; ++i)
      if (pids[i] >= 0)
        bulk_g2s(dst + (size_t)i * sub, C.pool + ((size_t)pids[i] * P.hkv + g) * (size_t)sub, (uint32_t)sub,
                 &sh.full[stg]);
  };
  if (tid == 0)
    for (int k = 0; k < kStages - 1 && k < nchunks; ++k) issue(k);

  float accv[VPL][CB][4];
#pragma unroll
  for (int p = 0; p < VPL; ++p)
#pragma unroll
    for (int c = 0; c < CB; ++c)
#pragma unroll
      for (int r = 0; r < 4; ++r) accv[p][c][r] = 0.f;

  for (int k = 0; k < nchunks; ++k) {
    __syncthreads();  // chunk k-1 fully consumed: its stage and sh.wsm may be rewritten
    if (tid == 0 && k + kStages - 1 < nchunks) issue(k + kStages - 1);
    const int stg = k % kStages;
    if (!mbar_wait_bounded(&sh.full[stg], (uint32_t)((k / kStages) & 1))) {
      atomicOr(&g_decode_err, TQ_DEVERR_TIMEOUT);
      sh.abort = 1;
    }
    __syncthreads();
    if (sh.abort) break;
    unsigned char* stbase = stage0 + (size_t)stg * kChunkPages * sub;

    // ---------------- key phase: warp w scores page w of the chunk
    const int pg = p0 + k * kChunkPages + warp;
    const bool pvalid = pg < p1 && sh.pvalid[stg][warp];
    unsigned char* pb = stbase + (size_t)warp * sub;
    float sc[2][2];
    {
      float accm[2][4], accq[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) accm[nt][r] = accq[nt][r] = 0.f;
      if (pvalid) {
        const uint32_t* kc = reinterpret_cast<const uint32_t*>(pb + P.off_kcodes);
        const uint32_t* ks = reinterpret_cast<const uint32_t*>(pb + P.off_ksigns);
        // plane words of token 8 nt + g8, words t4 * WPL + jw; inverted (bit set -> -1)
        uint32_t nwp[2][8][WPL];
        uint32_t nwq[2][WPL];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int tk = 8 * nt + g8;
#pragma unroll
          for (int jw = 0; jw < WPL; ++jw) {
            const int w = t4 * WPL + jw;
            const uint32_t sgn = kc[(0 * kPage + tk) * E + w];
            uint32_t mag[3] = {0u, 0u, 0u};
            for (int pl = 1; pl < P.kb; ++pl) mag[pl - 1] = kc[(pl * kPage + tk) * E + w];
#pragma unroll
            for (int S = 0; S < 8; ++S) {
              uint32_t wd = sgn;
              if (S & 1) wd ^= mag[0];
              if (S & 2) wd ^= mag[1];
              if (S & 4) wd ^= mag[2];
              nwp[nt][S][jw] = S < P.kp ? ~wd : 0u;
            }
            nwq[nt][jw] = P.kqjl ? ~ks[tk * E + w] : 0u;
          }
        }
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int jw = kk / 8, i0 = 2 * (kk % 8);
#pragma unroll
          for (int S = 0; S < 8; ++S) {
            if (S < P.kp) {
              const uint4 a = afr[(S * KS + kk) * 32 + lane];
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
                mma16816(accm[nt], a, pm1_pair(nwp[nt][S][jw], i0), pm1_pair(nwp[nt][S][jw], i0 + 1));
            }
          }
          if (P.kqjl) {
            const uint4 a = afr[(P.kp * KS + kk) * 32 + lane];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              mma16816(accq[nt], a, pm1_pair(nwq[nt][jw], i0), pm1_pair(nwq[nt][jw], i0 + 1));
          }
        }
      }
      const float* knorm = reinterpret_cast<const float*>(pb + P.off_knorm);
      const float* krn = reinterpret_cast<const float*>(pb + P.off_krnorm);
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * nt + 2 * t4 + e;
          const int tok = pg * kPage + t;
          const bool live = pvalid && g8 < G && tok < nc;
          float l = -INFINITY;
          if (live) {
            const float mse = accm[nt][e] + accm[nt][e + 2];
            const float qj = accq[nt][e] + accq[nt][e + 2];
            const float gm = P.kqjl ? krn[t] : 0.f;
            l = scale * knorm[t] * (mse * inv_sqrt_d + kappa * gm * qj);
            if (scores) scores[(head0 + g8) * (size_t)max_ctx + tok] = l;
          }
          sc[nt][e] = l;
          mx = fmaxf(mx, l);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (t4 == 0) sh.redm[warp][g8] = mx;
    }
    __syncthreads();
    if (tid < G) {
      float cm = sh.redm[0][tid];
#pragma unroll
      for (int w = 1; w < kChunkPages; ++w) cm = fmaxf(cm, sh.redm[w][tid]);
      const float mold = sh.mrun[tid];
      const float mnew = fmaxf(mold, cm);
      sh.alpha[tid] = mnew == -INFINITY ? 1.f : expf(mold - mnew);
      sh.mrun[tid] = mnew;
    }
    __syncthreads();
    {
      // weights of this warp's page: exp(l - m) * ||v|| / sqrt(d)
      const float* vnorm = reinterpret_cast<const float*>(pb + P.off_vnorm);
      const float m = g8 < G ? sh.mrun[g8] : 0.f;
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 8 * nt + 2 * t4 + e;
          float wgt = 0.f;
          if (sc[nt][e] != -INFINITY) {
            const float ex = expf(sc[nt][e] - m);
            ls += ex;
            wgt = ex * vnorm[t] * inv_sqrt_d;
          }
          if (g8 < G) sh.wsm[warp * kPage + t][g8] = wgt;
        }
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
      if (t4 == 0) sh.reds[warp][g8] = ls;
    }
    __syncthreads();
    if (tid < G) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kChunkPages; ++w) sum += sh.reds[w][tid];
      sh.lrun[tid] = sh.lrun[tid] * sh.alpha[tid] + sum;
    }
    // ---------------- value phase: warp w owns coordinates [w*CPW, (w+1)*CPW)
    {
      const float al = g8 < G ? sh.alpha[g8] : 1.f;
#pragma unroll
      for (int p = 0; p < VPL; ++p)
#pragma unroll
        for (int c = 0; c < CB; ++c)
#pragma unroll
          for (int r = 0; r < 4; ++r) accv[p][c][r] *= al;
#pragma unroll
      for (int jg = 0; jg < kChunkPages / 2; ++jg) {
        const unsigned char* pa = stbase + (size_t)(2 * jg) * sub;
        const unsigned char* pbb = stbase + (size_t)(2 * jg + 1) * sub;
        const uint16_t* va = reinterpret_cast<const uint16_t*>(pa + P.off_vcodes);
        const uint16_t* vbp = reinterpret_cast<const uint16_t*>(pbb + P.off_vcodes);
        // weights fragment for the two k-steps of this page pair: rows h (hi) / h + 8 (lo),
        // k-pair (2t, 2t+1) <-> token i of page A / page B with i = 8 ks + 2 t (+1 for k + 8)
        uint4 wf[2];
#pragma unroll
        for (int ksx = 0; ksx < 2; ++ksx) {
          const int i0 = 8 * ksx + 2 * t4, i1 = i0 + 1;
          const float wA0 = sh.wsm[(2 * jg) * kPage + i0][g8], wB0 = sh.wsm[(2 * jg + 1) * kPage + i0][g8];
          const float wA1 = sh.wsm[(2 * jg) * kPage + i1][g8], wB1 = sh.wsm[(2 * jg + 1) * kPage + i1][g8];
          __half hA0, lA0, hB0, lB0, hA1, lA1, hB1, lB1;
          split_f16(wA0, hA0, lA0);
          split_f16(wB0, hB0, lB0);
          split_f16(wA1, hA1, lA1);
          split_f16(wB1, hB1, lB1);
          wf[ksx].x = pack_h2(hA0, hB0);
          wf[ksx].y = pack_h2(lA0, lB0);
          wf[ksx].z = pack_h2(hA1, hB1);
          wf[ksx].w = pack_h2(lA1, lB1);
        }
#pragma unroll
        for (int cbk = 0; cbk < CB; ++cbk) {
          const int c = warp * CPW + cbk * 8 + g8;
          if (!VLUT) {
            const uint32_t u0 = (uint32_t)va[c] | ((uint32_t)vbp[c] << 16);
            uint32_t u1 = u0;
            if (P.vb == 2) u1 = u0 ^ ((uint32_t)va[D + c] | ((uint32_t)vbp[D + c] << 16));
            const uint32_t n0 = ~u0, n1 = ~u1;
#pragma unroll
            for (int ksx = 0; ksx < 2; ++ksx) {
              const int i0 = 8 * ksx + 2 * t4;
              mma16816(accv[0][cbk], wf[ksx], pm1_pair(n0, i0), pm1_pair(n0, i0 + 1));
              if (P.vb == 2) mma16816(accv[1][cbk], wf[ksx], pm1_pair(n1, i0), pm1_pair(n1, i0 + 1));
            }
          } else {
            uint32_t u[TQ_MAX_BITS];
#pragma unroll
            for (int p = 0; p < TQ_MAX_BITS; ++p)
              u[p] = p < P.vb ? ((uint32_t)va[p * D + c] | ((uint32_t)vbp[p * D + c] << 16)) : 0u;
#pragma unroll
            for (int ksx = 0; ksx < 2; ++ksx) {
              const int i0 = 8 * ksx + 2 * t4;
              uint32_t rA0 = 0, rB0 = 0, rA1 = 0, rB1 = 0;
#pragma unroll
              for (int p = 0; p < TQ_MAX_BITS; ++p) {
                rA0 |= ((u[p] >> i0) & 1u) << p;
                rB0 |= ((u[p] >> (i0 + 16)) & 1u) << p;
                rA1 |= ((u[p] >> (i0 + 1)) & 1u) << p;
                rB1 |= ((u[p] >> (i0 + 17)) & 1u) << p;
              }
              const uint32_t eA0 = sh.vlut[rA0], eB0 = sh.vlut[rB0], eA1 = sh.vlut[rA1], eB1 = sh.vlut[rB1];
              // hi halves -> plane 0, lo halves -> plane 1; pair = (token of page A, token of page B)
              mma16816(accv[0][cbk], wf[ksx], __byte_perm(eA0, eB0, 0x5410), __byte_perm(eA1, eB1, 0x5410));
              mma16816(accv[1][cbk], wf[ksx], __byte_perm(eA0, eB0, 0x7632), __byte_perm(eA1, eB1, 0x7632));
            }
          }
        }
      }
    }
  }
  __syncthreads();
  if (sh.abort) {
    // a bounded wait ran out: give the copies still in flight a second bounded
    // chance to land before the CTA's shared memory is released
    for (int k = 0; k < nchunks; ++k) (void)mbar_wait_bounded(&sh.full[k % kStages], (uint32_t)((k / kStages) & 1));
  }
  // partials: acc_rot[h][c] = sum over planes of coefficient x (hi-limb row + lo-limb row)
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  if (g8 < G) {
    const float c0 = VLUT ? 1.f : P.avw[0];
    const float c1 = VLUT ? 1.f : (P.vb == 2 ? P.avw[1] : 0.f);
#pragma unroll
    for (int cbk = 0; cbk < CB; ++cbk) {
      const int c = warp * CPW + cbk * 8 + 2 * t4;
      const float v0 = c0 * (accv[0][cbk][0] + accv[0][cbk][2]) + c1 * (accv[1][cbk][0] + accv[1][cbk][2]);
      const float v1 = c0 * (accv[0][cbk][1] + accv[0][cbk][3]) + c1 * (accv[1][cbk][1] + accv[1][cbk][3]);
      float* dst = acc + ((head0 + g8) * st + s) * D + c;
      dst[0] = v0;
      dst[1] = v1;
    }
  }
  if (tid < G) {
    ml[((head0 + tid) * st + s) * 2 + 0] = sh.mrun[tid];
    ml[((head0 + tid) * st + s) * 2 + 1] = sh.lrun[tid];
  }
}

// ------------------------------------------------------------------ combine

// One CTA per (query head, sequence): the split weights exp(m_s - M) are
// computed once into shared memory, then thread j sums the partials of
// coordinate j over the splits (coalesced across threads) and the rotated
// sum gets Pi_v^T once.
template <int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(const __grid_constant__ KParams P,
                                                           const unsigned char* ws, WsLayout L, float* out,
                                                           float* lse) {
  constexpr int E = D / 32;
  extern __shared__ __align__(16) float fsplit[];  // [st] split weights
  __shared__ float y[D];
  __shared__ float red[D / 32];
  __shared__ float Msh, Lsh;
  const int hq = blockIdx.x, b = blockIdx.y, j = threadIdx.x, lane = j & 31, warp = j >> 5;
  const int G = P.G, g = hq / G;
  const int st = L.n_comp_splits + 1;
  const size_t head = (size_t)b * P.hq + hq;
  const float* ml = reinterpret_cast<const float*>(ws + L.ml) + head * st * 2;
  const float* acc = reinterpret_cast<const float*>(ws + L.acc) + head * st * D;
  float m = -INFINITY;
  for (int k = j; k < st; k += D) m = fmaxf(m, ml[2 * k]);
  m = warp_max_f(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (j == 0) {
    float M = red[0];
    for (int w = 1; w < D / 32; ++w) M = fmaxf(M, red[w]);
    Msh = M;
  }
  __syncthreads();
  const float M = Msh;
  float lsum = 0.f;
  for (int k = j; k < st; k += D) {
    const float mk = ml[2 * k];
    const float f = (M == -INFINITY || mk == -INFINITY) ? 0.f : expf(mk - M);
    fsplit[k] = f;
    lsum += f * ml[2 * k + 1];
  }
  lsum = warp_sum_f(lsum);
  __syncthreads();
  if (lane == 0) red[warp] = lsum;
  __syncthreads();
  if (j == 0) {
    float s2 = 0.f;
    for (int w = 0; w < D / 32; ++w) s2 += red[w];
    Lsh = s2;
  }
  float rot = 0.f;
#pragma unroll 4
  for (int k = 0; k < st - 1; ++k) rot = fmaf(fsplit[k], acc[(size_t)k * D + j], rot);
  const float win = fsplit[st - 1] * acc[(size_t)(st - 1) * D + j];
  y[j] = rot;
  __syncthreads();
  const float* vrot = P.v_rot + (size_t)g * (P.kind == TQ_FWHT ? D : D * D);
  float o;
  if (P.kind == TQ_FWHT) {
    // Pi^T y = sigma * (H y) / sqrt(d)
    if (warp == 0) {
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = y[e * 32 + lane];
      warp_fwht<E>(a, lane);
      const float sc = rsqrtf((float)D);
      __syncwarp();
#pragma unroll
      for (int e = 0; e < E; ++e) y[e * 32 + lane] = a[e] * sc * __ldg(vrot + e * 32 + lane);
    }
    __syncthreads();
    o = y[j];
  } else {
    float a = 0.f;
#pragma unroll 8
    for (int jj = 0; jj < D; ++jj) a = fmaf(__ldg(vrot + (size_t)jj * D + j), y[jj], a);  // column j of Pi_v
    o = a;
  }
  const float Lsum = Lsh;
  const bool empty = M == -INFINITY || Lsum <= 0.f;
  out[head * D + j] = empty ? 0.f : (o + win) / Lsum;
  if (lse && j == 0) lse[head] = empty ? -INFINITY : M + logf(Lsum);
}

// ------------------------------------------------------------------ launcher

template <int D, bool VLUT>
static cudaError_t launch_mma(const KParams& P, const KCache& C, float scale, float* scores, unsigned char* ws,
                              const WsLayout& L, int max_ctx, cudaStream_t st) {
  const size_t dyn = L.afrag_bytes_per_head + (size_t)kStages * kChunkPages * P.sub_bytes;
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, VLUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)dyn);
  if (e != cudaSuccess) return e;
  dim3 grid(L.n_comp_splits, P.hkv, C.batch);
  decode_mma_kernel<D, VLUT><<<grid, kMmaThreads, dyn, st>>>(P, C, scale, scores, ws, L, max_ctx);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_decode_d(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                                   float* out, float* lse, float* scores, void* ws, const WsLayout& L, int max_ctx,
                                   cudaStream_t st) {
  unsigned char* w = reinterpret_cast<unsigned char*>(ws);
  cudaError_t e;
  const dim3 gh(P.hq, C.batch);
  decode_prologue_kernel<D><<<gh, D, 0, st>>>(P, q, dtype, w, L);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t wdyn = (size_t)std::max(1, C.ring) * TQ_MAX_GQA * sizeof(float);
  if (wdyn > 48 * 1024) {
    e = cudaFuncSetAttribute(decode_window_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wdyn);
    if (e != cudaSuccess) return e;
  }
  decode_window_kernel<D><<<dim3(P.hkv, C.batch), kWinThreads, wdyn, st>>>(P, C, q, dtype, scale, scores, w, L,
                                                                           max_ctx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = P.vb >= 3 ? launch_mma<D, true>(P, C, scale, scores, w, L, max_ctx, st)
                : launch_mma<D, false>(P, C, scale, scores, w, L, max_ctx, st);
  if (e != cudaSuccess) return e;
  const size_t cdyn = (size_t)(L.n_comp_splits + 1) * sizeof(float);
  if (cdyn > 48 * 1024) {
    e = cudaFuncSetAttribute(decode_combine_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cdyn);
    if (e != cudaSuccess) return e;
  }
  decode_combine_kernel<D><<<gh, D, cdyn, st>>>(P, w, L, out, lse);
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
