// Decode attention over the compressed paged cache (sm_103a).
//
// [Design study] §Transform placement: the query is moved into the rotated
// key basis once, scores are computed against the packed key codes, value
// pages are streamed after the softmax; §CPU and WASM kernel design: FP32
// score and output accumulators, value accumulation in the rotated value
// basis with ONE inverse transform per head.  [Reconstruction] §6: score
//   l = scale * n * ( <q', C[idx]> / sqrt(d) + sqrt(pi/2)/d * gamma * <q'', 2s - 1> ),
//   q' = Pi q, q'' = S q'.
// Keys with EDEN's unbiased scale or TurboVec's length-renormalized correction in
// place of the sketch ([Reconstruction] §10, §12) drop the second term and multiply the
// first by the stored scale s:  l = scale * n * s * <q', C[idx]> / sqrt(d).
//
// The two contractions of a decode step are dense products over the G query
// heads of a KV head:  scores[h, t] = sum_j Q[h, j] K_hat[t, j] and
// acc[h, j] = sum_t w[h, t] V_hat[t, j].  They run on the tensor cores
// (mma.m16n8k16, f16 operands, f32 accumulation) with operands that are
// EXACT in f16:
//   * a b-bit code with sign s and magnitude bits m has centroid
//     s * sum_S a_S prod_{i in S} (1 - 2 m_i) (Walsh expansion over the
//     magnitude bits), so the token side is a sum of +-1 "planes" whose
//     bit is s ^ parity(m & S); each f16 pair of an operand register comes
//     from one LOP3 on the packed word (or a copy shifted by 6 or 10): the
//     bit, kept at an exponent or sign position of 1.0 (2.0), reads as
//     base + b delta, the other operand carries x / delta, and the +-1
//     plane contracts to 2 D - K with a per-head constant K;
//   * the query side a_S q' (and q'') and the softmax weights are split into
//     f16 hi + lo limbs that occupy rows h and h + 8 of the 16-row tile
//     (G <= 8 heads), so the second limb costs no extra instruction;
//   * values with b >= 3 bits use f16 hi / lo limbs of the centroid itself
//     (two planes) read from a 16-entry table, instead of 2^(b-1) planes.
// Products are exact and accumulation is f32, so the scores carry ~2^-22
// relative query rounding instead of f16's 2^-11.
//
// Launches per call:
//   decode_prologue_kernel  grid (Hkv, ceil(batch G / 2), d / 64): q' = Pi q,
//                           q'' = S q' (64 rows of S per CTA) and the query
//                           rows of the score operands in mma fragment order;
//                           the decode kernel is launched as its programmatic
//                           dependent and starts streaming pages meanwhile.
//   decode_mma_kernel       grid (splits + 1, Hkv, batch): split-K over the page
//                           list.  Pages stream into shared memory with 1-D
//                           TMA bulk copies (cp.async.bulk + mbarrier, two or
//                           three stages of 8 pages); warp w scores page w of
//                           each 8-page chunk, then every warp accumulates
//                           values for its eighth of the coordinates.  The
//                           last split scans the float16 window (unrotated
//                           basis, CUDA cores) concurrently.
//   decode_combine_kernel   grid (Hq, batch): merges the partials in a fixed
//                           order, applies Pi_v^T once, adds the window part.
#include <math.h>

#include <algorithm>

#include "tq_device.cuh"
#include "tq_launch.h"
#include "tq_tile.cuh"

namespace tq {

__device__ unsigned int g_decode_err = 0;

#ifdef TQ_TEST_HOOKS
// Test build only: when set, the first chunk of every page split expects 16 bytes more than
// its copies deliver, so its barrier phase never completes and the bounded wait runs out.
__device__ int g_test_wait_fault = 0;
__device__ __forceinline__ uint32_t test_extra_tx(int k) { return (g_test_wait_fault && k == 0) ? 16u : 0u; }
#else
__device__ __forceinline__ uint32_t test_extra_tx(int) { return 0u; }
#endif

constexpr int kMmaThreads = 256;
constexpr int kMmaPages = kMmaThreads / 32;  // pages per chunk: one per warp in the key phase
constexpr int kStages = 3;
constexpr int kCombThreads = 256;
constexpr int kPrologueTile = 4;  // query vectors per prologue CTA: one wave of CTAs at the bench shapes
// Bounded mbarrier waits: at most kWaitLimit polls, each suspending at most kPollNs: about
// a second in the library; the test build (TQ_TEST_HOOKS) gives up after ~16 ms.
#ifdef TQ_TEST_HOOKS
constexpr unsigned kWaitLimit = 1u << 14;
#else
constexpr unsigned kWaitLimit = 1u << 20;
#endif
constexpr unsigned kPollNs = 1000;

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Resident decode CTAs per SM: three at d = 128 (80 registers), two at d = 256,
// whose larger register tiles would spill under the three-CTA cap.
__host__ __device__ constexpr int mma_ctas_per_sm(int d) { return d == 128 ? 3 : 2; }

// Query operand of the score products, per (sequence, kv head): units of one k-step
// (32 lanes x 16 bytes), plane S at units frag_plane_base(S) ..  Mixed-channel keys keep
// the planes that hold the wider codes' top bit (S >= kp / 2) for the first KS / 2 k-steps
// only: those cover the coordinates < d/2, the other coordinates' operand would be zero.
__host__ __device__ inline int frag_plane_base(const KParams& P, int S, int KS) {
  const int h = P.kp / 2;
  return (!P.ksplit || S < h) ? S * KS : h * KS + (S - h) * (KS / 2);
}
// Coordinate ca of A-fragment entry (k-step kk, lane t4, register r) and the bit ib of the B
// side's word it meets (ca + 16 meets bit ib + 16).  Lane t4 reads word t4 + 4 (kk / 8), bits
// 2 (kk mod 8) + (r >= 2): at d = 256 the first KS / 2 k-steps are the coordinates < d/2.  At
// d = 128 the planes of the wider codes' top bit (mixed-channel keys) cover words 0 and 1 in
// KS / 2 k-steps instead: lane t4 reads word t4 & 1 shifted right by 8 (t4 >> 1).
template <int D>
__host__ __device__ inline void frag_entry(bool half_plane, int kk, int t4, int r, int& ca, int& ib) {
  ib = 2 * (kk % 8) + (r >= 2 ? 1 : 0);
  if (D == 128 && half_plane) ca = 32 * (t4 & 1) + 8 * (t4 >> 1) + ib;
  else ca = 32 * (t4 + 4 * (kk / 8)) + ib;
}
static int key_frag_units(const KParams& P) {
  if (P.kivi) return 0;  // the KIVI kernel reads the query rows directly
  const int KS = P.d / 16;
  return P.ksplit ? frag_plane_base(P, P.kp, KS) : (P.kp + (P.kqjl == TQ_KEY_QJL ? 1 : 0)) * KS;
}

WsLayout decode_ws_layout(const KParams& P, int batch, int max_ctx, int n_splits, int num_sms) {
  WsLayout L{};
  const int max_pages = std::max(1, (max_ctx + kPage - 1) / kPage);
  int S = n_splits;
  if (S <= 0) {
    const int units = std::max(1, batch * P.hkv);
    // two waves of resident CTAs, or one wave where that would leave a split fewer than
    // four 8-page chunks (the per-CTA start-up would not amortise).  With a window every unit
    // also runs a window split, which holds a slot too: counting it keeps the grid from
    // spilling a few CTAs into a further wave (Qwen-like call: 18 + 1 splits a unit fill two
    // waves exactly and take 174 us, 19 + 1 take 199 us)
    const int cps = mma_ctas_per_sm(P.d);
    const int win = P.window > 0 ? 1 : 0;
    S = (2 * cps * num_sms + units - 1) / units - win;
    if (S < 1 || max_pages / S < 32) S = (cps * num_sms + units - 1) / units - win;
    S = std::max(1, std::min(S, (max_pages + 7) / 8));
  }
  S = std::min(S, max_pages);
  const int pps = (max_pages + S - 1) / S;
  S = (max_pages + pps - 1) / pps;
  L.n_comp_splits = S;
  L.pages_per_split = pps;
  const size_t heads = (size_t)batch * P.hq;
  const int st = S + 1;
  L.afrag_bytes_per_head = (size_t)key_frag_units(P) * 32 * 16;
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

// One-LOP3 +-1 planes.  An f16 pair whose halves are 1.0 (0x3C00; 2.0 for
// position 14) gets bit p of each half XORed in: p = 10..13 clear an
// exponent bit of 1.0 (0.5, 0.25, 2^-4, 2^-8), p = 14 clears 2.0 to 0, p = 15
// flips the sign.  A plane bit b then reads v = base_p + b delta_p; the other
// operand carries x / delta_p, so the product sums to sum x b plus a
// constant, and the +-1 plane (2 b - 1) contracts to 2 D - K with
// K = sum_k A_k (2 base_k + delta_k) over the operand's entries.
__host__ __device__ constexpr int xpos_key(int i) { return i >= 10 ? i : (i >= 4 ? i + 6 : i + 10); }
__host__ __device__ constexpr uint32_t xbase(int p) { return p == 14 ? 0x40004000u : 0x3C003C00u; }
__host__ __device__ inline float xdelta(int p) {
  return p == 10 ? -0.5f : p == 11 ? -0.75f : p == 12 ? -0.9375f : p == 13 ? -0.99609375f : -2.0f;
}
__host__ __device__ inline float xkfac(int p) { return 2.0f * (p == 14 ? 2.0f : 1.0f) + xdelta(p); }
// RN(1 / xdelta(p)) (the correctly rounded quotients: -2, -4/3, -16/15, -256/255, -1/2)
__host__ __device__ inline float xdelta_inv(int p) {
  return p == 10 ? -2.0f : p == 11 ? -1.33333337f : p == 12 ? -1.06666672f : p == 13 ? -1.00392163f : -0.5f;
}
// B register of key bit i (and i + 16) from the word's copies shifted by 0, 6 and 10;
// b1, b2 = xbase(10), xbase(14) in registers
__device__ __forceinline__ uint32_t xreg_key(uint32_t w0, uint32_t w6, uint32_t w10, int i, uint32_t b1, uint32_t b2) {
  const int p = xpos_key(i);
  const uint32_t src = i >= 10 ? w0 : (i >= 4 ? w6 : w10);
  return (src & (0x00010001u << p)) ^ (p == 14 ? b2 : b1);
}
// Token slot t = 4 t4 + 2 e + k of a page (lane t4, register e, k-step k of the value
// tiles): a lane's 32-bit plane word (page A's 16 slots low, page B's high) shifted left by
// 12 - 4 t4 puts its slots at f16 bit positions 12 + 2 e + k, i.e. 12..15.
__host__ __device__ constexpr int xpos_val(int t) { return 12 + (t & 3); }

// N adjacent floats (N = 2 or 4, 4N-byte aligned) in one global store.
template <int N>
__device__ __forceinline__ void vstore_f32(float* p, const float (&v)[N]) {
  if (N == 4) *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[N > 2 ? 2 : 0], v[N > 3 ? 3 : 0]);
  else *reinterpret_cast<float2*>(p) = make_float2(v[0], v[N > 1 ? 1 : 0]);
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
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(kPollNs)
      : "memory");
  return ok != 0;
}

// Bounded wait: false if the phase did not complete within kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (unsigned i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// After a bounded wait ran out (stopped at chunk kstop, the same in every thread): flag it,
// then give the copies still in flight (chunks kstop - 1 .. kstop + nst - 2) a second bounded
// chance to land before the CTA's shared memory is released.  The partials of such a split
// are not meaningful; the error word reports it.
// `ahead`: how many chunks beyond the one being consumed are issued (nst - 1, or nst - 2 where the
// previous chunk's stage is still read while the next key phase runs).
__device__ __forceinline__ void drain_after_timeout(uint64_t* full, bool timed_out, int kstop, int nchunks, int nst,
                                                    int ahead) {
  if (!__syncthreads_or(timed_out)) return;
  if (threadIdx.x == 0) atomicOr(&g_decode_err, TQ_DEVERR_TIMEOUT);
  const int last = min(kstop - 1 + ahead, nchunks - 1);
  for (int j = max(kstop - 1, 0); j <= last; ++j) (void)mbar_wait_bounded(&full[j % nst], (uint32_t)((j / nst) & 1));
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ prologue

// One CTA per (kv head g, tile of kPrologueTile query vectors of that head across the
// batch): q' = Pi_g q and q'' = S_g q' as tile products (each row of Pi_g and
// S_g is read once per tile), then every vector's rows of the query operand
// of the score products, in mma.m16n8k16 A-fragment order:
//   frag[plane][kk][lane] = 4 x f16x2, rows h_local (hi limb) and h_local + 8
//   (lo limb), k-pair (2t, 2t+1) <-> bits (i0, i0+16) and (2t+8, 2t+9) <->
//   (i0+1, i0+17) of plane word w = t + 4 (kk / 8), i0 = 2 (kk mod 8),
//   t = lane mod 4 (see frag_entry for the mixed-channel planes at d = 128).
//   Rows of absent heads (h_local >= G) are zero.
template <int D>
__global__ void __launch_bounds__(D) decode_prologue_kernel(const __grid_constant__ KParams P, const void* q,
                                                            int dtype, unsigned char* ws, WsLayout L, int batch) {
  constexpr int KS = D / 16;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TileSmem<D>& s = *reinterpret_cast<TileSmem<D>*>(smem_raw);
  const int g = blockIdx.x, z = blockIdx.z, j = threadIdx.x;
  // the decode kernel may start streaming its pages now; it waits for these
  // operands before its first score
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int G = P.G;
  const int n0 = blockIdx.y * kPrologueTile;
  const int nv = min(kPrologueTile, batch * G - n0);
  // the query first (the rotation needs it at once); the rows of S this thread multiplies do
  // not depend on it: their loads follow and land while the query is rotated
  float qv[kPrologueTile];
#pragma unroll
  for (int v = 0; v < kPrologueTile; ++v) {
    const int n = n0 + v, b = n / G, hl = n % G;
    qv[v] = (v < nv && j < P.dh) ? load_elem(q, dtype, (long long)((((size_t)b * P.hq + (size_t)g * G + hl)) * P.dh + j))
                                 : 0.f;  // zero-padded to D
  }
  constexpr int TPR = D / 64;  // threads per row of S: each CTA owns 64 rows (coordinates 64 z .. 64 z + 63)
  const bool dense_s = P.kqjl == TQ_KEY_QJL && !P.qjl_srht;
  // thread su of a row takes the float4 columns i4 * TPR + su: TPR neighbouring threads read
  // contiguous 16-byte pieces of S and of the query (no shared-memory bank conflicts)
  const int srow = 64 * z + j / TPR, su = j % TPR;
  float4 sreg[16];
  if (dense_s) {
    const float4* rp = reinterpret_cast<const float4*>(P.qjl_s + (size_t)g * D * D + (size_t)srow * D) + su;
#pragma unroll
    for (int i4 = 0; i4 < 16; ++i4) sreg[i4] = __ldg(rp + i4 * TPR);
  }
#pragma unroll
  for (int v = 0; v < kPrologueTile; ++v) s.x[v][j] = qv[v];
  if (j < kTile) s.inv[j] = P.kind == TQ_FWHT ? rsqrtf((float)D) : 1.0f;
  __syncthreads();
  rotate_tile<D, kPrologueTile>(s, nv, P.kind, P.k_rot + (size_t)g * (P.kind == TQ_FWHT ? D : D * D));
  if (P.kqjl == TQ_KEY_QJL && P.qjl_srht) {
    // q'' = H (sigma_S * q'), one warp per query vector (every CTA computes all d rows)
    constexpr int E = D / 32;
    const int lane = j & 31, warp = j >> 5;
    const float* sg = P.qjl_s + (size_t)g * D;
    for (int v = warp; v < nv; v += D / 32) {
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = s.x[v][e * 32 + lane] * __ldg(sg + e * 32 + lane);
      warp_wht<E>(a, lane);
#pragma unroll
      for (int e = 0; e < E; ++e) s.r[v][e * 32 + lane] = a[e];
    }
  } else if (dense_s) {
    // q'' rows of this CTA: TPR neighbouring threads per row, 64 inputs each (row segment in sreg)
    float acc[kPrologueTile];
#pragma unroll
    for (int v = 0; v < kPrologueTile; ++v) acc[v] = 0.f;
#pragma unroll
    for (int i4 = 0; i4 < 16; ++i4) {
      const float4 p = sreg[i4];
#pragma unroll
      for (int v = 0; v < kPrologueTile; ++v) {
        const float4 xv = *reinterpret_cast<const float4*>(&s.x[v][(i4 * TPR + su) * 4]);  // rows >= nv hold zeros
        acc[v] = fmaf(p.x, xv.x, fmaf(p.y, xv.y, fmaf(p.z, xv.z, fmaf(p.w, xv.w, acc[v]))));
      }
    }
#pragma unroll
    for (int v = 0; v < kPrologueTile; ++v) {
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], o);
      if (v < nv && su == 0) s.r[v][srow] = acc[v];
    }
  }
  __syncthreads();
  // fragment entries whose coordinate lies in this CTA's rows 64 z .. 64 z + 63 (the rows of S q'
  // it computed): words 2z and 2z + 1, i.e. k-steps 8 (z / 2) .. 8 (z / 2) + 7 of lanes
  // t4 = 2 (z mod 2) + {0, 1}, 64 entries a plane; the top-bit planes of mixed-channel keys only
  // where they are stored (coordinates < d/2)
  const int nplanes = P.kp + (P.kqjl == TQ_KEY_QJL ? 1 : 0);
  const int per_row = nplanes * 64;
  // the entries of all nv query vectors in one pass: vector v has per_row entries of its own
  // rows (lanes with lane / 4 == hl) and, for the sequence's first head, per_row of every row of
  // an absent head (zeroed)
  const int nabs = 8 - G;
  int ntot = 0;
  for (int v = 0; v < nv; ++v) ntot += per_row * (((n0 + v) % G == 0) ? 1 + nabs : 1);
  for (int idx = j; idx < ntot; idx += D) {
    int v = 0, rem = idx;
    for (;;) {  // the vector of entry idx (at most kPrologueTile steps)
      const int cnt = per_row * (((n0 + v) % G == 0) ? 1 + nabs : 1);
      if (rem < cnt) break;
      rem -= cnt;
      ++v;
    }
    const int n = n0 + v, b = n / G, hl = n % G;
    uint32_t* frag = reinterpret_cast<uint32_t*>(ws + L.afrag + ((size_t)b * P.hkv + g) * L.afrag_bytes_per_head);
    const int rowsel = rem / per_row, e = rem - rowsel * per_row;
    const int r = e & 3, pl = e >> 6, qe = e & 63;
    const bool half_plane = P.ksplit && pl >= P.kp / 2;
    int kk, t4;
    if (D == 128 && half_plane) {  // words 0 and 1 across all four lanes, 4 k-steps
      if (z != 0) continue;
      kk = qe >> 4;
      t4 = (qe >> 2) & 3;
    } else {
      if (half_plane && z >= 2) continue;  // d = 256: not stored beyond the first half
      kk = 8 * (z >> 1) + (qe >> 3);
      t4 = 2 * (z & 1) + ((qe >> 2) & 1);
    }
    int ca, ib;
    frag_entry<D>(half_plane, kk, t4, r, ca, ib);
    const int g8 = rowsel == 0 ? hl : (G - 1 + rowsel);
    uint32_t val = 0;
    if (rowsel == 0) {
      const int cb = ca + 16;
      float va, vb;
      if (pl < P.kp) {
        // mixed-channel keys: coordinates < d/2 follow the wider book
        const float a = ca < D / 2 ? P.akw_hi[pl] : P.akw[pl];
        va = a * s.x[v][ca];
        vb = a * s.x[v][cb];
      } else {
        va = s.r[v][ca];
        vb = s.r[v][cb];
      }
      const float rd = xdelta_inv(xpos_key(ib));  // the B side reads bit ib as base + b delta
      va *= rd;
      vb *= rd;
      __half ha, la, hb, lb;
      split_f16(va, ha, la);
      split_f16(vb, hb, lb);
      val = (r & 1) ? pack_h2(la, lb) : pack_h2(ha, hb);
    }
    frag[((frag_plane_base(P, pl, KS) + kk) * 32 + g8 * 4 + t4) * 4 + r] = val;
  }
}

// ------------------------------------------------------------------ window (CUDA cores)

// The float16 window of one (kv head, sequence), run by the last split of the
// decode grid (concurrently with the page splits): chunks of 16 tokens are
// staged in shared memory with 16-byte loads; scores for the G heads (one
// warp per token, unrotated basis), an online softmax per head, and the
// weighted sum of the values (thread per coordinate).
template <int D>
__device__ void window_split(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                             float* scores, unsigned char* ws, const WsLayout& L, int max_ctx, int g, int b,
                             unsigned char* smem) {
  constexpr int E = D / 32, NT = kMmaThreads;
  constexpr int NG = NT / D, TG = kPage / NG;  // value phase: token groups
  __half* kst = reinterpret_cast<__half*>(smem);                     // [16][D]
  __half* vst = kst + kPage * D;                                     // [16][D]
  float* qs = reinterpret_cast<float*>(vst + kPage * D);             // [G][D]
  float* sc = qs + TQ_MAX_GQA * D;                                   // [16][8]
  float* st_m = sc + kPage * TQ_MAX_GQA;                             // [8] running max
  float* st_l = st_m + TQ_MAX_GQA;                                   // [8] running sum
  float* st_a = st_l + TQ_MAX_GQA;                                   // [8] rescale
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = P.G;
  const int st = L.n_comp_splits + 1;
  const size_t head0 = (size_t)b * P.hq + (size_t)g * G;
  const int cb = C.parent ? C.parent[b] : b;  // cache row of (virtual) sequence b
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
  for (int i = tid; i < G * D; i += NT) {
    const int h = i / D, j = i % D;
    qs[i] = j < P.dh ? load_elem(q, dtype, (long long)((head0 + h) * P.dh + j)) : 0.f;  // zero-padded to D
  }
  if (tid < TQ_MAX_GQA) {
    st_m[tid] = -INFINITY;
    st_l[tid] = 0.f;
  }
  const int cj = tid % D, tg = tid / D;
  float acc[TQ_MAX_GQA];
#pragma unroll
  for (int h = 0; h < TQ_MAX_GQA; ++h) acc[h] = 0.f;
  const size_t ring0 = ((size_t)cb * P.hkv + g) * (size_t)C.ring;
  for (int c0 = 0; c0 < nw; c0 += kPage) {
    __syncthreads();
    constexpr int V16 = D / 8;  // 16-byte vectors per row
    for (int i = tid; i < 2 * kPage * V16; i += NT) {
      const int which = i / (kPage * V16), t = (i / V16) % kPage, v8 = i % V16;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (c0 + t < nw) {
        const __half* src = (which ? C.win_v : C.win_k) + (ring0 + (size_t)((nc + c0 + t) % C.ring)) * D;
        val = reinterpret_cast<const uint4*>(src)[v8];
      }
      reinterpret_cast<uint4*>(which ? vst : kst)[t * V16 + v8] = val;
    }
    __syncthreads();
    for (int t = warp; t < kPage; t += NT / 32) {
      const bool live = c0 + t < nw;
      float kv[E];
#pragma unroll
      for (int e = 0; e < E; ++e) kv[e] = __half2float(kst[t * D + e * 32 + lane]);
      for (int h = 0; h < G; ++h) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) a = fmaf(qs[h * D + e * 32 + lane], kv[e], a);
        a = warp_sum_f(a);
        if (lane == 0) {
          sc[t * TQ_MAX_GQA + h] = live ? scale * a : -INFINITY;
          if (scores && live) scores[(head0 + h) * (size_t)max_ctx + nc + c0 + t] = scale * a;
        }
      }
    }
    __syncthreads();
    if (warp < G && lane < kPage) {  // warp h updates head h over the 16 tokens
      const int h = warp;
      const float l = sc[lane * TQ_MAX_GQA + h];
      float mx = l;
      for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0x0000ffffu, mx, o));
      const float mnew = fmaxf(st_m[h], mx);
      const float e = (l == -INFINITY) ? 0.f : expf(l - mnew);
      float sm = e;
      for (int o = 8; o > 0; o >>= 1) sm += __shfl_xor_sync(0x0000ffffu, sm, o);
      sc[lane * TQ_MAX_GQA + h] = e;
      __syncwarp(0x0000ffffu);
      if (lane == 0) {
        const float a = (mnew == -INFINITY) ? 1.f : expf(st_m[h] - mnew);
        st_a[h] = a;
        st_l[h] = st_l[h] * a + sm;
        if (mnew != -INFINITY) st_m[h] = mnew;
      }
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < TQ_MAX_GQA; ++h) {
      if (h < G) {
        float a = acc[h] * st_a[h];
#pragma unroll
        for (int tt = 0; tt < TG; ++tt) {
          const int t = tg * TG + tt;
          a = fmaf(sc[t * TQ_MAX_GQA + h], __half2float(vst[t * D + cj]), a);
        }
        acc[h] = a;
      }
    }
  }
  __syncthreads();
  // reduce token groups through the (now free) staging buffer
  float* red = reinterpret_cast<float*>(smem);  // [NT][8]
#pragma unroll
  for (int h = 0; h < TQ_MAX_GQA; ++h) red[tid * TQ_MAX_GQA + h] = acc[h];
  __syncthreads();
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  float* accw = reinterpret_cast<float*>(ws + L.acc);
  if (tid < D) {
    for (int h = 0; h < G; ++h) {
      float v = 0.f;
#pragma unroll
      for (int gr = 0; gr < NG; ++gr) v += red[(gr * D + tid) * TQ_MAX_GQA + h];
      accw[((head0 + h) * st + (st - 1)) * D + tid] = v;
    }
  }
  if (tid < G) {
    ml[((head0 + tid) * st + (st - 1)) * 2 + 0] = st_m[tid];
    ml[((head0 + tid) * st + (st - 1)) * 2 + 1] = st_l[tid];
  }
}

// Shared memory the window split needs (staging, query, scores, state, reduction).
static size_t window_smem_bytes(int d) {
  const size_t stage = 2 * (size_t)kPage * d * sizeof(__half) + (size_t)TQ_MAX_GQA * d * sizeof(float) +
                       (size_t)(kPage + 3) * TQ_MAX_GQA * sizeof(float);
  const size_t red = (size_t)kMmaThreads * TQ_MAX_GQA * sizeof(float);
  return std::max(stage, red);
}

// ------------------------------------------------------------------ compressed pages (tensor cores)

constexpr int kPidCache = 1024;  // block-table entries of a split staged in shared memory

struct MmaShared {
  uint64_t full[kStages];
  uint4 wf[2][kMmaPages / 2][2][32];  // softmax weights in mma A-fragment order, per page pair (chunk parity)
  float redm[kMmaPages][TQ_MAX_GQA];  // per-warp chunk maxima
  float lsum[kMmaPages][TQ_MAX_GQA];  // per-warp softmax denominators
  float mfin[TQ_MAX_GQA];
  float kvsum[kMmaPages][TQ_MAX_GQA];  // per-warp sums of the value operand's constant
  float kcon[2][TQ_MAX_GQA];           // constant K of the key operand: MSE planes, QJL plane
  uint32_t vlut[16];  // values with b >= 3: raw sign-magnitude bits -> (hi, lo) f16 of the centroid
};

// KMIX: the layer uses mixed-channel keys or byte key norms (compiled out otherwise).
// KPF > 0: TurboQuant_prod keys (QJL sketch) with KPF Walsh planes, fixed at compile time;
// with KMIX, KPF = 8: mixed-channel keys of 3 + 1 bits (eight planes for the wider half, the
// key correction read at run time)
// (kp = 2 for 2-bit codes, 4 for 3-bit), values of 2 bits or more (2-bit planes when !VLUT);
// KPF = 0 reads the plane count, correction and value bits at run time.
template <int D, bool VLUT, bool KMIX, int KPF>
__global__ void __launch_bounds__(kMmaThreads, mma_ctas_per_sm(D)) decode_mma_kernel(const __grid_constant__ KParams P,
                                                                 const __grid_constant__ KCache C, const void* q,
                                                                 int dtype, float scale, float* scores,
                                                                 unsigned char* ws, WsLayout L, int max_ctx,
                                                                 int nst) {
  constexpr int E = D / 32, WPL = D / 128, KS = D / 16;
  constexpr int NW = kMmaThreads / 32;  // warps = pages per chunk
  constexpr int CPW = D / NW;           // value coordinates per warp
  constexpr int CB = CPW / 8;           // n-tiles per value plane per warp
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ MmaShared sh;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  // the combine kernel may be scheduled once every CTA of this grid has started; it waits
  // for the whole grid before it reads the partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (s == L.n_comp_splits) {  // the float16 window runs as the last split
    window_split<D>(P, C, q, dtype, scale, scores, ws, L, max_ctx, g, b, dyn);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, t4 = lane & 3;
  const int G = P.G;
  const int st = L.n_comp_splits + 1;
  const size_t head0 = (size_t)b * P.hq + (size_t)g * G;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float kappa = sqrtf(1.57079632679489662f) / (float)D;
  const int sub = P.sub_bytes;
  const uint32_t xb1 = P.xb1, xb2 = P.xb2;
  const bool ksplit = KMIX && P.ksplit, knu8 = KMIX && P.knu8;
  const int kp = KPF > 0 ? KPF : P.kp;
  const int kqjl = (KPF > 0 && !KMIX) ? (int)TQ_KEY_QJL : P.kqjl;
  const int kbits = KPF > 0 ? (KPF == 2 ? 2 : 3) : P.kb;
  constexpr int kUnrollS = (KPF > 0 && !KMIX) ? KPF : (KMIX && KPF > 0 ? 2 : 1);
  auto pbase = [&](int S) { return ksplit ? frag_plane_base(P, S, KS) : S * KS; };
  const bool vb2 = (KPF > 0 && !KMIX && !VLUT) ? true : P.vb == 2;  // the QJL variants carry 2-bit planes

  // shared memory: query fragments | page stages | page ids of this split
  uint4* afr = reinterpret_cast<uint4*>(dyn);                                  // [planes][KS][32]
  unsigned char* stage0 = dyn + L.afrag_bytes_per_head;                        // [nst][NW][sub]
  long long* pids = reinterpret_cast<long long*>(stage0 + (size_t)nst * NW * sub);  // [<= kPidCache]

  const int cb = C.parent ? C.parent[b] : b;  // cache row of (virtual) sequence b
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
  const int npg = max(0, p1 - p0);
  const int nchunks = (npg + NW - 1) / NW;
  const int ncache = min(npg, kPidCache);

  for (int i = tid; i < ncache; i += kMmaThreads) {
    long long pid = C.block_table[(size_t)cb * C.max_pages + p0 + i];
    if (pid < 0 || pid >= C.n_pages) {
      atomicOr(&g_decode_err, TQ_DEVERR_PAGE_INDEX);
      pid = -1;
    }
    pids[i] = pid;
  }
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
    for (int i = 0; i < kStages; ++i) mbar_init(&sh.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  auto page_id = [&](int i) -> long long {  // i = page index within the split
    if (i >= npg) return -1;
    if (i < ncache) return pids[i];
    long long pid = C.block_table[(size_t)cb * C.max_pages + p0 + i];
    if (pid < 0 || pid >= C.n_pages) {
      atomicOr(&g_decode_err, TQ_DEVERR_PAGE_INDEX);
      pid = -1;
    }
    return pid;
  };
  // producer (warp 0, lane i < NW handles page i): chunk k = split pages
  // NW k .. NW k + NW - 1 into stage k % nst
  auto issue = [&](int k) {
    const int stg = k % nst;
    const long long pid = lane < NW ? page_id(k * NW + lane) : -1;
    const unsigned valid = __ballot_sync(0xffffffffu, pid >= 0);
    if (lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&sh.full[stg], (uint32_t)__popc(valid) * (uint32_t)sub + test_extra_tx(k));
    }
    __syncwarp();
    if (pid >= 0)
      bulk_g2s(stage0 + ((size_t)stg * NW + lane) * sub, C.pool + ((size_t)pid * P.hkv + g) * (size_t)sub,
               (uint32_t)sub, &sh.full[stg]);
  };
  if (warp == 0)
    for (int k = 0; k < nst - 2 && k < nchunks; ++k) issue(k);
  // the query fragments come from the prologue kernel (launched just before, with
  // this grid allowed to start early): wait for it, then stage them; the first
  // page copies are already in flight
  asm volatile("griddepcontrol.wait;" ::: "memory");
  {
    const uint4* src = reinterpret_cast<const uint4*>(ws + L.afrag + ((size_t)b * P.hkv + g) * L.afrag_bytes_per_head);
    for (int i = tid; i < (int)(L.afrag_bytes_per_head / 16); i += kMmaThreads) afr[i] = src[i];
  }
  __syncthreads();
  if (warp < G) {
    // K of head `warp`: its A-fragment rows (lanes 4 warp .. 4 warp + 3) over all stored planes and
    // k-blocks; register r of block kk pairs with key bit 2 (kk mod 8) + (r >= 2)
    const int nplanes = kp + (kqjl == TQ_KEY_QJL ? 1 : 0);
    float km = 0.f, kq = 0.f;
    for (int it = lane; it < nplanes * KS * 4; it += 32) {
      const int pl = it / (KS * 4), kk = (it / 4) % KS, t4i = it % 4;
      if (ksplit && pl >= kp / 2 && kk >= KS / 2) continue;  // not stored: zero operand
      const uint4 a = afr[(pbase(pl) + kk) * 32 + warp * 4 + t4i];
      const uint32_t rr[4] = {a.x, a.y, a.z, a.w};
      float sum = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float f = xkfac(xpos_key(2 * (kk % 8) + (r >= 2 ? 1 : 0)));
        sum += f * (__half2float(__ushort_as_half((unsigned short)(rr[r] & 0xffffu))) +
                    __half2float(__ushort_as_half((unsigned short)(rr[r] >> 16))));
      }
      if (pl < kp) km += sum;
      else kq += sum;
    }
    km = warp_sum_f(km);
    kq = warp_sum_f(kq);
    if (lane == 0) {
      sh.kcon[0][warp] = km;
      sh.kcon[1][warp] = kq;
    }
  }

  float accv[2][CB][4];
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int c = 0; c < CB; ++c)
#pragma unroll
      for (int r = 0; r < 4; ++r) accv[p][c][r] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // softmax state of head g8 (identical across warps for m)
  float kv_run = 0.f;                     // this lane's share of the value operand's constant K
  // value phase of chunk kc (its stage, weights buffer kc & 1): warp w owns coordinates
  // [w*CPW, (w+1)*CPW); runs at the top of iteration kc + 1, overlapping that chunk's key phase
  auto value_phase = [&](int kc) {
    unsigned char* stbase = stage0 + (size_t)(kc % nst) * NW * sub;
    const uint4(&wfb)[kMmaPages / 2][2][32] = sh.wf[kc & 1];
#pragma unroll 1
    for (int jg = 0; jg < NW / 2; ++jg) {
      const uint16_t* va = reinterpret_cast<const uint16_t*>(stbase + (size_t)(2 * jg) * sub + P.off_vcodes);
      const uint16_t* vbp = reinterpret_cast<const uint16_t*>(stbase + (size_t)(2 * jg + 1) * sub + P.off_vcodes);
      const uint4 wf0 = wfb[jg][0][lane], wf1 = wfb[jg][1][lane];
      if (!VLUT) {
        // plane words: page A's 16 slots in bits 0..15, page B's in 16..31 (one byte permute per
        // word); column g8 of n-tile cbk is coordinate warp * CPW + g8 * CB + cbk, so a lane's CB
        // entries of a plane are adjacent (one vector load per page and plane).  Shifted left by
        // 12 - 4 t4, the lane's slots 4 t4 + 2 e + k sit at bit 12 + 2 e + k of each half: operand
        // register e of k-step k is one LOP3 (mask, then XOR into 1.0 / 2.0)
        uint32_t u0[CB], u1[CB];
        {
          const int c0 = warp * CPW + g8 * CB;
          if constexpr (CB == 4) {
            const uint2 a0 = *reinterpret_cast<const uint2*>(va + c0), b0 = *reinterpret_cast<const uint2*>(vbp + c0);
            u0[0] = __byte_perm(a0.x, b0.x, 0x5410);
            u0[1] = __byte_perm(a0.x, b0.x, 0x7632);
            u0[CB > 2 ? 2 : 0] = __byte_perm(a0.y, b0.y, 0x5410);
            u0[CB > 3 ? 3 : 0] = __byte_perm(a0.y, b0.y, 0x7632);
            if (vb2) {
              const uint2 a1 = *reinterpret_cast<const uint2*>(va + D + c0),
                          b1 = *reinterpret_cast<const uint2*>(vbp + D + c0);
              u1[0] = __byte_perm(a1.x, b1.x, 0x5410);
              u1[1] = __byte_perm(a1.x, b1.x, 0x7632);
              u1[CB > 2 ? 2 : 0] = __byte_perm(a1.y, b1.y, 0x5410);
              u1[CB > 3 ? 3 : 0] = __byte_perm(a1.y, b1.y, 0x7632);
            }
          } else {
            const uint32_t a0 = *reinterpret_cast<const uint32_t*>(va + c0),
                           b0 = *reinterpret_cast<const uint32_t*>(vbp + c0);
            u0[0] = __byte_perm(a0, b0, 0x5410);
            u0[CB > 1 ? 1 : 0] = __byte_perm(a0, b0, 0x7632);
            if (vb2) {
              const uint32_t a1 = *reinterpret_cast<const uint32_t*>(va + D + c0),
                             b1 = *reinterpret_cast<const uint32_t*>(vbp + D + c0);
              u1[0] = __byte_perm(a1, b1, 0x5410);
              u1[CB > 1 ? 1 : 0] = __byte_perm(a1, b1, 0x7632);
            }
          }
        }
        const int vsh = 12 - 4 * t4;
#pragma unroll
        for (int cbk = 0; cbk < CB; ++cbk) {
          const uint32_t x0 = u0[cbk] << vsh;
          const uint32_t xm = vb2 ? (u1[cbk] << vsh) : 0u;
#pragma unroll
          for (int ksx = 0; ksx < 2; ++ksx) {
            const uint4 wfk = ksx ? wf1 : wf0;
            const int pA = 12 + ksx, pB = 14 + ksx;  // register e = 0, 1
            const uint32_t mA = 0x00010001u << pA, mB = 0x00010001u << pB;
            const uint32_t bA = (x0 & mA) ^ (pA == 14 ? xb2 : xb1), bB = (x0 & mB) ^ (pB == 14 ? xb2 : xb1);
            mma16816(accv[0][cbk], wfk, bA, bB);
            if (vb2) mma16816(accv[1][cbk], wfk, bA ^ (xm & mA), bB ^ (xm & mB));  // Walsh plane sign ^ magnitude
          }
        }
      } else {
#pragma unroll
        for (int cbk = 0; cbk < CB; ++cbk) {
          const int c = warp * CPW + g8 * CB + cbk;
          // the table index of each of this lane's slots 4 t4 .. 4 t4 + 3 (pages A and B) as a
          // nibble: slot j of page A at nibble j, of page B at nibble 4 + j, plane p at bit p
          uint32_t iw = 0;
#pragma unroll
          for (int p = 0; p < TQ_MAX_BITS; ++p) {
            if (p < P.vb) {
              const uint32_t u = (uint32_t)va[p * D + c] | ((uint32_t)vbp[p * D + c] << 16);
              const uint32_t x = (u >> (4 * t4)) & 0x000F000Fu;
              iw |= ((x | (x << 3) | (x << 6) | (x << 9)) & 0x11111111u) << p;
            }
          }
#pragma unroll
          for (int ksx = 0; ksx < 2; ++ksx) {
            // slots 4 t4 + ksx (register e = 0) and 4 t4 + 2 + ksx (e = 1)
            const uint32_t rA0 = (iw >> (4 * ksx)) & 15u, rB0 = (iw >> (16 + 4 * ksx)) & 15u;
            const uint32_t rA1 = (iw >> (8 + 4 * ksx)) & 15u, rB1 = (iw >> (24 + 4 * ksx)) & 15u;
            const uint32_t eA0 = sh.vlut[rA0], eB0 = sh.vlut[rB0], eA1 = sh.vlut[rA1], eB1 = sh.vlut[rB1];
            const uint4 wfk = ksx ? wf1 : wf0;
            // hi halves -> plane 0, lo halves -> plane 1; pair = (token of page A, token of page B)
            mma16816(accv[0][cbk], wfk, __byte_perm(eA0, eB0, 0x5410), __byte_perm(eA1, eB1, 0x5410));
            mma16816(accv[1][cbk], wfk, __byte_perm(eA0, eB0, 0x7632), __byte_perm(eA1, eB1, 0x7632));
          }
        }
      }
    }
  };
  bool timed_out = false;
  int kstop = nchunks;  // chunks consumed

  for (int k = 0; k <= nchunks; ++k) {
    // softmax of chunk k-1 done (its weights are in sh.wf[(k-1) & 1]).  A wait that ran out
    // stops the split here, for every thread alike (no new copies into unfinished phases)
    if (__syncthreads_or(timed_out)) {
      kstop = k;
      break;
    }
    // chunk k + nst - 2 goes to the stage of chunk k - 2 (its values were accumulated in the
    // previous iteration): stages k - 1 (values below) and k (keys below) stay untouched
    if (warp == 0 && k < nchunks && k + nst - 2 < nchunks) issue(k + nst - 2);
    if (k > 0) value_phase(k - 1);
    if (k == nchunks) break;
    const int stg = k % nst;
    if (!mbar_wait_bounded(&sh.full[stg], (uint32_t)((k / nst) & 1))) timed_out = true;
    unsigned char* stbase = stage0 + (size_t)stg * NW * sub;

    // ---------------- key phase: warp w scores page w of the chunk
    const int pi = k * NW + warp;
    const bool pvalid = pi < npg && page_id(pi) >= 0;
    const int pg = p0 + pi;
    const unsigned char* pb = stbase + (size_t)warp * sub;
    float sc[2][2];
    {
      float accm[2][2][4], accq[2][2][4];  // [kk parity][n-tile][frag]
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) accm[x][nt][r] = accq[x][nt][r] = 0.f;
      if (pvalid) {
        const uint32_t* kc = reinterpret_cast<const uint32_t*>(pb + P.off_kcodes);
        const uint32_t* kx = reinterpret_cast<const uint32_t*>(pb + P.off_kx);
        // raw words of token 8 nt + g8: word t4 + 4 jw (jw = kk / 8); mixed-channel keys: magnitude
        // plane kb (the wider codes' top bit) exists for words < E / 2 only
        uint32_t rs[2][WPL], rm[3][2][WPL];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int jw = 0; jw < WPL; ++jw) {
            const int tk = 2 * g8 + nt, w = t4 + 4 * jw;
            rs[nt][jw] = kc[tk * E + w];
#pragma unroll
            for (int m = 0; m < 3; ++m)
              rm[m][nt][jw] = (m + 1 < kbits)                                 ? kc[((m + 1) * kPage + tk) * E + w]
                              : (ksplit && m + 1 == kbits && w < E / 2) ? kx[tk * (E / 2) + w]
                                                                          : 0u;
          }
        // planes over all k-steps; mixed-channel keys: the planes holding the top bit follow
        const int s_full = ksplit ? kp / 2 : kp;
#pragma unroll kUnrollS
        for (int S = 0; S < s_full; ++S) {
          uint32_t w0[2][WPL], w6[2][WPL], w10[2][WPL];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int jw = 0; jw < WPL; ++jw) {
              w0[nt][jw] = rs[nt][jw] ^ ((S & 1) ? rm[0][nt][jw] : 0u) ^ ((S & 2) ? rm[1][nt][jw] : 0u) ^
                           ((S & 4) ? rm[2][nt][jw] : 0u);
              w6[nt][jw] = w0[nt][jw] << 6;
              w10[nt][jw] = w0[nt][jw] << 10;
            }
          const uint4* ap = afr + (size_t)pbase(S) * 32 + lane;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint4 a = ap[kk * 32];
            const int jw = kk / 8, i0 = 2 * (kk % 8);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              mma16816(accm[kk & 1][nt], a, xreg_key(w0[nt][jw], w6[nt][jw], w10[nt][jw], i0, xb1, xb2),
                       xreg_key(w0[nt][jw], w6[nt][jw], w10[nt][jw], i0 + 1, xb1, xb2));
          }
        }
        if (ksplit) {
          // the planes with the top bit over the coordinates < d/2 only (KS / 2 k-steps)
          uint32_t hs[2], hm[3][2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            if (D == 256) {  // words t4 < E / 2: the jw = 0 words already loaded
              hs[nt] = rs[nt][0];
#pragma unroll
              for (int m = 0; m < 3; ++m) hm[m][nt] = rm[m][nt][0];
            } else {  // d = 128: word t4 & 1 shifted right by 8 (t4 >> 1)
              const int tk = 2 * g8 + nt, w = t4 & 1, sh = 8 * (t4 >> 1);
              hs[nt] = kc[tk * E + w] >> sh;
#pragma unroll
              for (int m = 0; m < 3; ++m)
                hm[m][nt] = ((m + 1 < kbits) ? kc[((m + 1) * kPage + tk) * E + w]
                                             : (m + 1 == kbits) ? kx[tk * (E / 2) + w] : 0u) >> sh;
            }
          }
#pragma unroll kUnrollS
          for (int S = kp / 2; S < kp; ++S) {
            uint32_t w0[2], w6[2], w10[2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              w0[nt] = hs[nt] ^ ((S & 1) ? hm[0][nt] : 0u) ^ ((S & 2) ? hm[1][nt] : 0u) ^ ((S & 4) ? hm[2][nt] : 0u);
              w6[nt] = w0[nt] << 6;
              w10[nt] = w0[nt] << 10;
            }
            const uint4* ap = afr + (size_t)frag_plane_base(P, S, KS) * 32 + lane;
#pragma unroll
            for (int kk = 0; kk < KS / 2; ++kk) {
              const uint4 a = ap[kk * 32];
              const int i0 = 2 * (kk % 8);
#pragma unroll
              for (int nt = 0; nt < 2; ++nt)
                mma16816(accm[kk & 1][nt], a, xreg_key(w0[nt], w6[nt], w10[nt], i0, xb1, xb2),
                         xreg_key(w0[nt], w6[nt], w10[nt], i0 + 1, xb1, xb2));
            }
          }
        }
        if (kqjl == TQ_KEY_QJL) {
          const uint32_t* ks = reinterpret_cast<const uint32_t*>(pb + P.off_ksigns);
          uint32_t q0[2][WPL], q6[2][WPL], q10[2][WPL];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int jw = 0; jw < WPL; ++jw) {
              q0[nt][jw] = ks[(2 * g8 + nt) * E + t4 + 4 * jw];
              q6[nt][jw] = q0[nt][jw] << 6;
              q10[nt][jw] = q0[nt][jw] << 10;
            }
          const uint4* ap = afr + (size_t)kp * KS * 32 + lane;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const uint4 a = ap[kk * 32];
            const int jw = kk / 8, i0 = 2 * (kk % 8);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              mma16816(accq[kk & 1][nt], a, xreg_key(q0[nt][jw], q6[nt][jw], q10[nt][jw], i0, xb1, xb2),
                       xreg_key(q0[nt][jw], q6[nt][jw], q10[nt][jw], i0 + 1, xb1, xb2));
          }
        }
      }
      const float* knorm = reinterpret_cast<const float*>(pb + P.off_knorm);  // or bytes (knu8)
      const float* krn = reinterpret_cast<const float*>(pb + P.off_krnorm);
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 4 * t4 + 2 * e + nt;  // column 2 t4 + e of n-tile nt (column g of n-tile nt is token 2 g + nt)
          const int tok = pg * kPage + t;
          const bool live = pvalid && g8 < G && tok < nc;
          float l = -INFINITY;
          if (live) {
            // +-1 plane sums from the operand sums: 2 D - K
            const float mse =
                2.f * (accm[0][nt][e] + accm[0][nt][e + 2] + accm[1][nt][e] + accm[1][nt][e + 2]) - sh.kcon[0][g8];
            const float qj = kqjl == TQ_KEY_QJL
                                 ? 2.f * (accq[0][nt][e] + accq[0][nt][e + 2] + accq[1][nt][e] + accq[1][nt][e + 2]) -
                                       sh.kcon[1][g8]
                                 : 0.f;
            // QJL: gamma times the sketch term; EDEN / renormalized keys: the scale s on the code's term
            const float gm = kqjl == TQ_KEY_QJL ? krn[t] : 0.f;
            const float sk = kqjl >= TQ_KEY_EDEN ? krn[t] : 1.f;
            const float kn = knu8 ? norm_u8_decode(pb[P.off_knorm + t], P) : knorm[t];
            l = scale * kn * (sk * (mse * inv_sqrt_d) + kappa * gm * qj);
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
    // ---------------- online softmax: every lane tracks the state of head g8
    float alpha = 1.f;
    {
      float cm = sh.redm[0][g8];
#pragma unroll
      for (int w = 1; w < NW; ++w) cm = fmaxf(cm, sh.redm[w][g8]);
      const float mnew = fmaxf(m_run, cm);
      if (mnew != -INFINITY) {
        alpha = expf(m_run - mnew);
        m_run = mnew;
      }
      // weights of this warp's page, written in A-fragment order of its page pair:
      // token t = 4 t4 + 2 e + nt -> k-step nt, lane (g8, t4), component 2 e (hi) / 2 e + 1 (lo),
      // half = page parity within the pair
      const float* vnorm = reinterpret_cast<const float*>(pb + P.off_vnorm);
      uint16_t* wfh = reinterpret_cast<uint16_t*>(&sh.wf[k & 1][warp >> 1][0][0]);
      float ls = 0.f, kvs = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 4 * t4 + 2 * e + nt;
          float wgt = 0.f;
          if (sc[nt][e] != -INFINITY) {
            const float ex = expf(sc[nt][e] - m_run);
            ls += ex;
            wgt = ex * vnorm[t] * inv_sqrt_d;
          }
          // +-1 value planes read slot t as base + b delta: the weight carries 1 / delta
          const int xp = xpos_val(t);
          if (!VLUT) wgt *= 1.0f / xdelta(xp);
          __half hi, lo;
          split_f16(wgt, hi, lo);
          if (!VLUT) kvs += (__half2float(hi) + __half2float(lo)) * xkfac(xp);
          uint16_t* dst = wfh + ((nt * 32 + lane) * 4 + 2 * e) * 2 + (warp & 1);
          dst[0] = __half_as_ushort(hi);
          dst[2] = __half_as_ushort(lo);
        }
      l_run = l_run * alpha + ls;
      kv_run = kv_run * alpha + kvs;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int p = 0; p < 2; ++p)
#pragma unroll
          for (int c = 0; c < CB; ++c)
#pragma unroll
            for (int r = 0; r < 4; ++r) accv[p][c][r] *= alpha;
      }
    }
  }
  drain_after_timeout(sh.full, timed_out, kstop, nchunks, nst, nst - 2);
  // ---- partials
  float ls = l_run, kvl = kv_run;
  ls += __shfl_xor_sync(0xffffffffu, ls, 1);
  ls += __shfl_xor_sync(0xffffffffu, ls, 2);
  kvl += __shfl_xor_sync(0xffffffffu, kvl, 1);
  kvl += __shfl_xor_sync(0xffffffffu, kvl, 2);
  if (t4 == 0) {
    sh.lsum[warp][g8] = ls;
    sh.kvsum[warp][g8] = kvl;
  }
  if (warp == 0 && t4 == 0) sh.mfin[g8] = m_run;
  __syncthreads();
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  if (g8 < G) {
    // acc_rot[h][c] = sum over planes of coefficient x (hi-limb row + lo-limb row)
    const float c0 = VLUT ? 1.f : P.avw[0];
    const float c1 = VLUT ? 1.f : (vb2 ? P.avw[1] : 0.f);
    // +-1 value planes: 2 D - K with K summed over every warp's tokens (the LUT limbs need no correction)
    float kv = 0.f;
    if (!VLUT) {
#pragma unroll
      for (int w = 0; w < NW; ++w) kv += sh.kvsum[w][g8];
    }
    const float pm = VLUT ? 1.f : 2.f;
    // columns 2 t4 and 2 t4 + 1 of n-tile cbk are coordinates warp * CPW + (2 t4) CB + cbk and
    // warp * CPW + (2 t4 + 1) CB + cbk: CB adjacent coordinates each, one vector store apiece
    float v0[CB], v1[CB];
#pragma unroll
    for (int cbk = 0; cbk < CB; ++cbk) {
      v0[cbk] = c0 * (pm * (accv[0][cbk][0] + accv[0][cbk][2]) - kv) +
                c1 * (pm * (accv[1][cbk][0] + accv[1][cbk][2]) - kv);
      v1[cbk] = c0 * (pm * (accv[0][cbk][1] + accv[0][cbk][3]) - kv) +
                c1 * (pm * (accv[1][cbk][1] + accv[1][cbk][3]) - kv);
    }
    float* dst = acc + ((head0 + g8) * st + s) * D + warp * CPW + 2 * t4 * CB;
    vstore_f32<CB>(dst, v0);
    vstore_f32<CB>(dst + CB, v1);
  }
  if (tid < G) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) l += sh.lsum[w][tid];
    ml[((head0 + tid) * st + s) * 2 + 0] = sh.mfin[tid];
    ml[((head0 + tid) * st + s) * 2 + 1] = l;
  }
}

// ------------------------------------------------------------------ combine

// One CTA per (query head, sequence): the split weights exp(m_s - M) are
// computed once into shared memory; the partial accumulators are summed by
// SG groups of threads (each group takes every SG-th split, float4 per
// thread, coalesced), the groups are reduced in shared memory, and the
// rotated sum gets Pi_v^T once.
template <int D>
__global__ void __launch_bounds__(kCombThreads) decode_combine_kernel(const __grid_constant__ KParams P,
                                                                      const unsigned char* ws, WsLayout L,
                                                                      float* out, float* lse) {
  constexpr int E = D / 32, TPR = D / 4, SG = kCombThreads / TPR;
  extern __shared__ __align__(16) float fsplit[];  // [st] split weights
  __shared__ __align__(16) float part[SG][D];
  __shared__ float y[D];
  __shared__ float red[kCombThreads / 32];
  __shared__ float Msh, Lsh;
  const int hq = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = P.G, g = hq / G;
  // launched as a programmatic dependent of the decode kernel: wait for all of its partials
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int st = L.n_comp_splits + 1;
  const size_t head = (size_t)b * P.hq + hq;
  const float* ml = reinterpret_cast<const float*>(ws + L.ml) + head * st * 2;
  const float* acc = reinterpret_cast<const float*>(ws + L.acc) + head * st * D;
  // the first kPre partial rows of this thread's split group are loaded up front, together with
  // the split maxima (one memory round trip instead of three)
  constexpr int kPre = 8;
  const int sg = tid / TPR, c4 = tid % TPR;
  float4 pre[kPre];
#pragma unroll
  for (int r = 0; r < kPre; ++r) {
    const int k = sg + r * SG;
    pre[r] = k < st - 1 ? reinterpret_cast<const float4*>(acc + (size_t)k * D)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY;
  for (int k = tid; k < st; k += kCombThreads) m = fmaxf(m, ml[2 * k]);
  m = warp_max_f(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (tid == 0) {
    float M = red[0];
    for (int w = 1; w < kCombThreads / 32; ++w) M = fmaxf(M, red[w]);
    Msh = M;
  }
  __syncthreads();
  const float M = Msh;
  float lsum = 0.f;
  for (int k = tid; k < st; k += kCombThreads) {
    const float mk = ml[2 * k];
    const float f = (M == -INFINITY || mk == -INFINITY) ? 0.f : expf(mk - M);
    fsplit[k] = f;
    lsum += f * ml[2 * k + 1];
  }
  lsum = warp_sum_f(lsum);
  __syncthreads();
  if (lane == 0) red[warp] = lsum;
  __syncthreads();
  if (tid == 0) {
    float s2 = 0.f;
    for (int w = 0; w < kCombThreads / 32; ++w) s2 += red[w];
    Lsh = s2;
  }
  // compressed splits 0 .. st-2: group sg sums splits sg, sg + SG, ... in a fixed order
  {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
      const int k = sg + r * SG;
      if (k < st - 1) {
        const float f = fsplit[k];
        a.x = fmaf(f, pre[r].x, a.x);
        a.y = fmaf(f, pre[r].y, a.y);
        a.z = fmaf(f, pre[r].z, a.z);
        a.w = fmaf(f, pre[r].w, a.w);
      }
    }
#pragma unroll 4
    for (int k = sg + kPre * SG; k < st - 1; k += SG) {
      const float f = fsplit[k];
      const float4 v = reinterpret_cast<const float4*>(acc + (size_t)k * D)[c4];
      a.x = fmaf(f, v.x, a.x);
      a.y = fmaf(f, v.y, a.y);
      a.z = fmaf(f, v.z, a.z);
      a.w = fmaf(f, v.w, a.w);
    }
    reinterpret_cast<float4*>(part[sg])[c4] = a;
  }
  __syncthreads();
  for (int j = tid; j < D; j += kCombThreads) {
    float r = 0.f;
#pragma unroll
    for (int sg = 0; sg < SG; ++sg) r += part[sg][j];
    y[j] = r;
  }
  __syncthreads();
  const float* vrot = P.v_rot + (size_t)g * (P.kind == TQ_FWHT ? D : D * D);
  if (P.kivi) {
    // values were accumulated in the original basis: no inverse rotation
  } else if (P.kind == TQ_FWHT) {
    // Pi^T y = sigma * (H y) / sqrt(d)
    if (warp == 0) {
      float a[E];
#pragma unroll
      for (int e = 0; e < E; ++e) a[e] = y[e * 32 + lane];
      warp_wht<E>(a, lane);
      const float sc = rsqrtf((float)D);
      __syncwarp();
#pragma unroll
      for (int e = 0; e < E; ++e) y[e * 32 + lane] = a[e] * sc * __ldg(vrot + e * 32 + lane);
    }
    __syncthreads();
  } else {
    float o = 0.f;
    if (tid < D) {
#pragma unroll 8
      for (int jj = 0; jj < D; ++jj) o = fmaf(__ldg(vrot + (size_t)jj * D + tid), y[jj], o);  // column of Pi_v
    }
    __syncthreads();
    if (tid < D) y[tid] = o;
    __syncthreads();
  }
  const float Lsum = Lsh;
  const bool empty = M == -INFINITY || Lsum <= 0.f;
  const float fw = fsplit[st - 1];
  for (int j = tid; j < D; j += kCombThreads) {
    const float win = fw * acc[(size_t)(st - 1) * D + j];
    if (j < P.dh) out[head * P.dh + j] = empty ? 0.f : (y[j] + win) / Lsum;
  }
  if (lse && tid == 0) lse[head] = empty ? -INFINITY : M + logf(Lsum);
}

// ------------------------------------------------------------------ KIVI control arm (tensor cores)

#include "tq_kivi_mma.cuh"
#include "tq_prefill_mma.cuh"

// ------------------------------------------------------------------ launcher

template <int D, bool VLUT, bool KMIX, int KPF>
static cudaError_t launch_mma(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                              float* scores, unsigned char* ws, const WsLayout& L, int max_ctx, cudaStream_t st) {
  const size_t pid_bytes = (size_t)std::min(L.pages_per_split, kPidCache) * sizeof(long long);
  const size_t stage_bytes = (size_t)kMmaPages * P.sub_bytes;
  int nst = kStages;
  size_t dyn = L.afrag_bytes_per_head + nst * stage_bytes + pid_bytes;
  if (dyn > (mma_ctas_per_sm(D) == 3 ? 72 : 110) * 1024) {  // keep the resident CTAs where the pages are large
    nst = 2;
    dyn = L.afrag_bytes_per_head + nst * stage_bytes + pid_bytes;
  }
  dyn = std::max(dyn, window_smem_bytes(D));
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, VLUT, KMIX, KPF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)dyn);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the grid may start while the prologue runs
  // (it waits on it with griddepcontrol.wait before reading the query fragments)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.n_comp_splits + 1, P.hkv, C.batch);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, VLUT, KMIX, KPF>, P, C, q, dtype, scale, scores, ws, L, max_ctx, nst);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int KB, int VB>
static cudaError_t launch_kivi(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                               float* scores, unsigned char* ws, const WsLayout& L, int max_ctx, cudaStream_t st) {
  const size_t pid_bytes = (size_t)std::min(L.pages_per_split, kPidCache) * sizeof(long long);
  const size_t stage_bytes = (size_t)kMmaPages * P.sub_bytes;
  const size_t head_bytes = (size_t)(D / 16) * 32 * sizeof(uint4) + (size_t)TQ_MAX_GQA * D * sizeof(float);
  int nst = kStages;
  size_t dyn = head_bytes + nst * stage_bytes + pid_bytes;
  if (dyn > 100 * 1024) {  // two resident CTAs
    nst = 2;
    dyn = head_bytes + nst * stage_bytes + pid_bytes;
  }
  dyn = std::max(dyn, window_smem_bytes(D));
  cudaError_t e = cudaFuncSetAttribute(kivi_mma_kernel<D, KB, VB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)dyn);
  if (e != cudaSuccess) return e;
  const dim3 grid(L.n_comp_splits + 1, P.hkv, C.batch);
  kivi_mma_kernel<D, KB, VB><<<grid, kMmaThreads, dyn, st>>>(P, C, q, dtype, scale, scores, ws, L, max_ctx, nst);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_kivi_bits(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                                    float* scores, unsigned char* ws, const WsLayout& L, int max_ctx, cudaStream_t st) {
  if (P.kb == 2 && P.vb == 2) return launch_kivi<D, 2, 2>(P, C, q, dtype, scale, scores, ws, L, max_ctx, st);
  if (P.kb == 2 && P.vb == 4) return launch_kivi<D, 2, 4>(P, C, q, dtype, scale, scores, ws, L, max_ctx, st);
  if (P.kb == 4 && P.vb == 2) return launch_kivi<D, 4, 2>(P, C, q, dtype, scale, scores, ws, L, max_ctx, st);
  return launch_kivi<D, 4, 4>(P, C, q, dtype, scale, scores, ws, L, max_ctx, st);
}

template <int D>
static cudaError_t launch_decode_d(const KParams& P, const KCache& C, const void* q, int dtype, float scale,
                                   float* out, float* lse, float* scores, void* ws, const WsLayout& L, int max_ctx,
                                   cudaStream_t st) {
  unsigned char* w = reinterpret_cast<unsigned char*>(ws);
  if (P.kivi) {  // no query transform: pages, window, then the merge
    cudaError_t e = launch_kivi_bits<D>(P, C, q, dtype, scale, scores, w, L, max_ctx, st);
    if (e != cudaSuccess) return e;
    const size_t cdyn = (size_t)(L.n_comp_splits + 1) * sizeof(float);
    if (cdyn > 48 * 1024) {
      e = cudaFuncSetAttribute(decode_combine_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cdyn);
      if (e != cudaSuccess) return e;
    }
    decode_combine_kernel<D><<<dim3(P.hq, C.batch), kCombThreads, cdyn, st>>>(P, w, L, out, lse);
    return cudaGetLastError();
  }
  const size_t tsm = sizeof(TileSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(decode_prologue_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsm);
  if (e != cudaSuccess) return e;
  const dim3 gp(P.hkv, (C.batch * P.G + kPrologueTile - 1) / kPrologueTile, D / 64);
  decode_prologue_kernel<D><<<gp, D, tsm, st>>>(P, q, dtype, w, L, C.batch);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const bool kmix = P.ksplit || P.knu8;
  // TurboQuant_prod keys with 2 or 3 code bits: plane count and sketch fixed at compile time
  const int kpf = (!kmix && P.kqjl == TQ_KEY_QJL && (P.kp == 2 || P.kp == 4) && P.vb >= 2) ? P.kp : 0;
  // mixed-channel keys of 3 + 1 bits: eight Walsh planes fixed at compile time
  const bool kmix8 = kmix && P.ksplit && P.kp == 8 && P.kb == 3;
  if (P.vb >= 3)
    e = kmix8      ? launch_mma<D, true, true, 8>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
        : kmix     ? launch_mma<D, true, true, 0>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
        : kpf == 2 ? launch_mma<D, true, false, 2>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
        : kpf == 4 ? launch_mma<D, true, false, 4>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
                   : launch_mma<D, true, false, 0>(P, C, q, dtype, scale, scores, w, L, max_ctx, st);
  else
    e = kmix8      ? launch_mma<D, false, true, 8>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
        : kmix     ? launch_mma<D, false, true, 0>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
        : kpf == 2 ? launch_mma<D, false, false, 2>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
        : kpf == 4 ? launch_mma<D, false, false, 4>(P, C, q, dtype, scale, scores, w, L, max_ctx, st)
                   : launch_mma<D, false, false, 0>(P, C, q, dtype, scale, scores, w, L, max_ctx, st);
  if (e != cudaSuccess) return e;
  const size_t cdyn = (size_t)(L.n_comp_splits + 1) * sizeof(float);
  if (cdyn > 48 * 1024) {
    e = cudaFuncSetAttribute(decode_combine_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cdyn);
    if (e != cudaSuccess) return e;
  }
  // programmatic dependent launch: scheduled while the decode grid drains
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.hq, C.batch);
  cfg.blockDim = dim3(kCombThreads);
  cfg.dynamicSmemBytes = cdyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, P, (const unsigned char*)w, L, out, lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_decode(const KParams& P, const KCache& C, const void* q, int dtype, float scale, float* out,
                          float* lse, float* scores, void* ws, const WsLayout& L, int max_ctx, cudaStream_t st) {
  if (P.d == 128) return launch_decode_d<128>(P, C, q, dtype, scale, out, lse, scores, ws, L, max_ctx, st);
  return launch_decode_d<256>(P, C, q, dtype, scale, out, lse, scores, ws, L, max_ctx, st);
}

// ------------------------------------------------------------------ prefill tiles

bool prefill_tiles_ok(const KParams& P) {
  if (P.kivi || P.ksplit || P.knu8 || P.kqjl != TQ_KEY_QJL || (P.kp != 2 && P.kp != 4) || P.vb < 2) return false;
  if (P.d != 128 && P.d != 256) return false;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    optin = 232448;  // sm_103a: 227 KB a block
  }
  const size_t afr = (size_t)kPfTiles * (P.kp + 1) * (P.d / 16) * 32 * 16;
  const size_t need = afr + (size_t)2 * kPfWarps * P.sub_bytes + (size_t)kPfPidCache * sizeof(long long) + sizeof(PfShared);
  return need <= (size_t)optin;
}

// Compressed splits of the tile path: the split count (1..8, at least 32 pages a split) whose
// CTAs (one per SM) fill their last wave best, a point of fill outweighing one more split.
int prefill_tile_splits(const KParams& P, int batch, int n_query, int max_ctx, int num_sms) {
  const long long ups = ((long long)n_query * P.G + kPfRows - 1) / kPfRows;
  const long long units = std::max(1LL, (long long)batch * P.hkv * ups);
  const int max_pages = std::max(1, (max_ctx + kPage - 1) / kPage);
  int best = 1;
  double best_eff = -1.0;
  for (int S = 1; S <= 8; ++S) {
    if (S > 1 && max_pages / S < 32) break;
    const double w = (double)(units * S) / std::max(1, num_sms);
    const double eff = w / ceil(w) - 0.01 * (S - 1);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = S;
    }
  }
  return best;
}

template <int D, bool VLUT, int KPF>
static cudaError_t launch_tiles(const KParams& P, const KCache& C, int n_query, int batch, float scale,
                                unsigned char* ws, const WsLayout& L, int max_ctx, cudaStream_t st) {
  const int ups = (n_query * P.G + kPfRows - 1) / kPfRows;
  const size_t pid_bytes = (size_t)std::min(L.pages_per_split, kPfPidCache) * sizeof(long long);
  const size_t afr = (size_t)kPfTiles * L.afrag_bytes_per_head;
  const size_t stage_bytes = (size_t)kPfWarps * P.sub_bytes;
  int dev = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  int nst = kStages;
  size_t dyn = afr + nst * stage_bytes + pid_bytes;
  if (dyn + sizeof(PfShared) > (size_t)optin) {
    nst = 2;
    dyn = afr + nst * stage_bytes + pid_bytes;
  }
  e = cudaFuncSetAttribute(prefill_tiles_kernel<D, VLUT, KPF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
  if (e != cudaSuccess) return e;
  // programmatic dependent of the prologue: pages stream while it runs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.n_comp_splits, P.hkv, batch * ups);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, prefill_tiles_kernel<D, VLUT, KPF>, P, C, n_query, ups, scale, ws, L, max_ctx, nst);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_prefill_tiles_d(const KParams& P, const KCache& V, int n_query, int batch, const void* q,
                                          int dtype, float scale, float* out, float* lse, unsigned char* w,
                                          const WsLayout& L, int max_ctx, cudaStream_t st) {
  const int nv = V.batch;
  const size_t tsm = sizeof(TileSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(decode_prologue_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tsm);
  if (e != cudaSuccess) return e;
  const dim3 gp(P.hkv, (nv * P.G + kPrologueTile - 1) / kPrologueTile, D / 64);
  decode_prologue_kernel<D><<<gp, D, tsm, st>>>(P, q, dtype, w, L, nv);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (P.vb >= 3)
    e = P.kp == 2 ? launch_tiles<D, true, 2>(P, V, n_query, batch, scale, w, L, max_ctx, st)
                  : launch_tiles<D, true, 4>(P, V, n_query, batch, scale, w, L, max_ctx, st);
  else
    e = P.kp == 2 ? launch_tiles<D, false, 2>(P, V, n_query, batch, scale, w, L, max_ctx, st)
                  : launch_tiles<D, false, 4>(P, V, n_query, batch, scale, w, L, max_ctx, st);
  if (e != cudaSuccess) return e;
  const size_t wdyn = window_smem_bytes(D);
  if (wdyn > 48 * 1024) {
    e = cudaFuncSetAttribute(prefill_attn_window_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wdyn);
    if (e != cudaSuccess) return e;
  }
  prefill_attn_window_kernel<D><<<dim3(P.hkv, nv), kMmaThreads, wdyn, st>>>(P, V, q, dtype, scale, w, L, max_ctx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t cdyn = (size_t)(L.n_comp_splits + 1) * sizeof(float);
  if (cdyn > 48 * 1024) {
    e = cudaFuncSetAttribute(decode_combine_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cdyn);
    if (e != cudaSuccess) return e;
  }
  decode_combine_kernel<D><<<dim3(P.hq, nv), kCombThreads, cdyn, st>>>(P, w, L, out, lse);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tiles(const KParams& P, const KCache& V, int n_query, int batch, const void* q, int dtype,
                                 float scale, float* out, float* lse, void* ws, const WsLayout& L, int max_ctx,
                                 cudaStream_t st) {
  unsigned char* w = reinterpret_cast<unsigned char*>(ws);
  if (P.d == 128)
    return launch_prefill_tiles_d<128>(P, V, n_query, batch, q, dtype, scale, out, lse, w, L, max_ctx, st);
  return launch_prefill_tiles_d<256>(P, V, n_query, batch, q, dtype, scale, out, lse, w, L, max_ctx, st);
}

__global__ void prefill_virtual_kernel(const __grid_constant__ KCache C, int n_query, int32_t* seq_v,
                                       int32_t* nc_v, int32_t* parent) {
  const long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (v >= (long long)C.batch * n_query) return;
  const int b = (int)(v / n_query), i = (int)(v % n_query);
  const int T = C.seq_len[b], nc = C.n_compressed[b];
  int tv = T - n_query + i + 1;  // query i sees positions 0 .. T - n_query + i
  if (T < n_query || nc < 0 || nc > T) {
    if (i == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
    tv = max(tv, 0);
  }
  seq_v[v] = tv;
  nc_v[v] = min(max(nc, 0), tv);
  parent[v] = b;
}

cudaError_t launch_prefill_virtual(const KCache& C, int n_query, int32_t* seq_v, int32_t* nc_v, int32_t* parent,
                                   cudaStream_t st) {
  const long long n = (long long)C.batch * n_query;
  prefill_virtual_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(C, n_query, seq_v, nc_v, parent);
  return cudaGetLastError();
}

#ifdef TQ_TEST_HOOKS
cudaError_t set_test_wait_fault(int on) { return cudaMemcpyToSymbol(g_test_wait_fault, &on, sizeof(int)); }
#endif

cudaError_t read_clear_decode_error(unsigned* bits) {
  unsigned zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_decode_err, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_decode_err, &zero, sizeof(unsigned));
}

}  // namespace tq
