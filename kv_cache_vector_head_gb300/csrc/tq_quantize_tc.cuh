// Bulk quantize of d = 128 bf16 keys with the FWHT rotation and the QJL
// sketch: both products on tcgen05, one vector per thread in the epilogues.
//
// [Reconstruction] §5 Steps 1-5 (norm, rotation, code, residual, QJL signs)
// and §6 (the stored record); [Design study] §CPU and WASM kernel design
// ("Append-time key kernel").  Same decisions as quantize_keys_tc_kernel and
// quantize_warp_kernel (fp32 values of the same accuracy, the exact cell
// table for the codes, the certified sketch bound with an fp32 recompute),
// laid out for the 5th-generation tensor cores:
//
//   * a CTA holds two independent groups of 8 warps; a group owns a tile of
//     128 tokens of one kv head per pass: M = 128 rows of every UMMA, one
//     row per TMEM lane.  While one group waits for its loads or its tensor
//     work, the other computes;
//   * the tile's bf16 rows are copied (cp.async) into the UMMA A layout and
//     rotated by ONE product Z = X (H diag(sigma))^T on tcgen05 (kind::f16,
//     bf16 operands; +-1 and bf16 values are exact, accumulation in fp32)
//     into tensor memory;
//   * the epilogue thread of row r and column half h reads 64 rotated
//     coordinates with tcgen05.ld, codes them through the cell table,
//     packs its plane words with byte permutes (no shuffles) and writes the
//     residual's f16 hi / lo limbs back over the consumed input tile, which
//     is then the A operand of S r (three limb products, as in
//     quantize_keys_tc_kernel);
//   * the sketch epilogue reads one row's 64 sketch coordinates per thread,
//     takes the signs and recomputes in fp32 the entries within the
//     certified bound.
// Norms are taken from the bf16 inputs (exact squares, balanced fp32 trees)
// while the rotation runs.
//
// Values and keys without the sketch stay on quantize_warp_kernel, whose
// register-resident FWHT needs no tensor-memory round trip.
//
// Requirements checked by the launcher: d = 128, FWHT, keys with the QJL
// sketch, head_dim <= 128 and a multiple of 8, bf16 16-byte aligned input,
// antisymmetric tables, a cell table scale J that fits the shared memory,
// flat outputs.
#pragma once

#include "tq_quantize_mma.cuh"

namespace tq {
namespace wq {

constexpr int kBtWarps = 16;  // two groups of 8
constexpr int kBtThreads = 32 * kBtWarps;
constexpr size_t kBtTile = kUmmaTile;  // 128 x 128 16-bit operand: 32 KB

struct BtShared {
  float part[2][2][128];  // [group][column half][row]: partial sums (norm, then the residual's)
  uint64_t mbar[2][2];    // [group][product]
  uint32_t tmem;
  float smax;
};

// Operand bytes: the rotation B tile, S hi / lo, and per group the input tile, then the
// residual limbs (two tiles)
__host__ __device__ constexpr size_t bt_smem_bytes(int J) {
  return 3 * kBtTile + 2 * 2 * kBtTile + sizeof(BtShared) + lut_bytes(J, false);
}

// Named barrier of one group (barrier 1 + G, n threads).
__device__ __forceinline__ void bt_bar(int G, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + G), "r"(n) : "memory");
}

// Named barrier of one group that also ORs a flag over its threads (every thread of the
// group leaves with the same value).
__device__ __forceinline__ bool bt_bar_or(int G, int n, bool v) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.s32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((int)v), "r"(1 + G), "r"(n)
      : "memory");
  return r != 0;
}

// Bounded wait on a tcgen05 commit barrier: at most 2^20 polls, each suspending the thread
// for up to 1 us (it resumes when the phase completes); false when it ran out (about a second).
__device__ __forceinline__ bool bt_wait(uint64_t* bar, uint32_t phase) {
  uint32_t done = 0;
  for (unsigned it = 0; it < (1u << 20) && !done; ++it)
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(phase), "n"(1000));
  return done != 0;
}

__device__ __forceinline__ void bt_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
        "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
        "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void bt_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(accum));
}

// Balanced sum of 32 values.
__device__ __forceinline__ float tree32(const float (&a)[32]) {
  float b[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) b[i] = a[2 * i] + a[2 * i + 1];
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) b[i] = b[2 * i] + b[2 * i + 1];
  return b[0];
}

// Plane words of 32 coordinates from four byte accumulators (byte p of acc[k]: plane p of
// coordinates 8k .. 8k + 7): word p = byte p of acc[0..3].
__device__ __forceinline__ void planes_of(const uint32_t (&acc)[4], uint32_t (&w)[4]) {
  const uint32_t lo01 = __byte_perm(acc[0], acc[1], 0x5140), hi01 = __byte_perm(acc[0], acc[1], 0x7362);
  const uint32_t lo23 = __byte_perm(acc[2], acc[3], 0x5140), hi23 = __byte_perm(acc[2], acc[3], 0x7362);
  w[0] = __byte_perm(lo01, lo23, 0x5410);
  w[1] = __byte_perm(lo01, lo23, 0x7632);
  w[2] = __byte_perm(hi01, hi23, 0x5410);
  w[3] = __byte_perm(hi01, hi23, 0x7632);
}

// grid (x, Hkv): CTA (x, h) takes tiles x * 2 + G (+ 2 * gridDim.x) of kv head h.
template <int BITS>
__global__ void __launch_bounds__(kBtThreads, 1)
    quantize_bt_kernel(const __grid_constant__ KParams P, const __nv_bfloat16* __restrict__ x, long long n_vec,
                       uint32_t* __restrict__ codes, uint32_t* __restrict__ signs, float* __restrict__ norms,
                       float* __restrict__ rnorms, int lut_j) {
  constexpr int GT = 256;  // threads per group
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* Brot = smem_raw;
  unsigned char* Bhi = smem_raw + kBtTile;
  unsigned char* Blo = Bhi + kBtTile;
  unsigned char* buf0 = smem_raw + 3 * kBtTile;
  BtShared& ts = *reinterpret_cast<BtShared*>(buf0 + 2 * 2 * kBtTile);
  unsigned char* lut_at = reinterpret_cast<unsigned char*>(&ts) + sizeof(BtShared);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = warp >> 3, wg = warp & 7, gt = tid & 255;  // group, warp in group, thread in group
  const int sp = wg & 3, h = wg >> 2;                      // TMEM sub-partition (rows), column half
  const int head = blockIdx.y;
  const float* sig = P.k_rot + (size_t)head * D;
  const float* S = P.qjl_s + (size_t)head * (P.qjl_srht ? D : D * D);
  unsigned char* buf = buf0 + (size_t)G * 2 * kBtTile;

  build_code_lut<BITS, false>(lut_at, lut_j, P.kt, P.kc, tid, kBtThreads);
  if (warp == 0) {  // tensor memory: per group the rotation and the sketch accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ts.tmem)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int g = 0; g < 2; ++g)
      for (int k = 0; k < 2; ++k) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&ts.mbar[g][k])), "r"(1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // ---- per-CTA constants: B[n][k] = H[n][k] sigma_k (bf16 +-1); S limbs; max ||S_c||
  for (int i = tid; i < D * (D / 8); i += kBtThreads) {
    const int n = i >> 4, k0 = 8 * (i & 15);
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t hw[2];
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const int k = k0 + 2 * e + f;
        const bool neg = (__ldg(sig + k) < 0.f) != (bool)(__popc(n & k) & 1);
        hw[f] = neg ? 0xBF80u : 0x3F80u;
      }
      w[e] = hw[0] | (hw[1] << 16);
    }
    *reinterpret_cast<uint4*>(Brot + umma_off(n, k0)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  {
    for (int i = tid; i < D * (D / 4); i += kBtThreads) {
      const int c = i >> 5, k0 = 4 * (i & 31);
      float4 sv;
      if (P.qjl_srht) {  // S[c][k] = (-1)^popcount(c & k) sigma_S[k], exact in f16 (lo limb 0)
        const float4 sg = __ldg(reinterpret_cast<const float4*>(S) + (i & 31));
        sv = make_float4((__popc(c & k0) & 1) ? -sg.x : sg.x, (__popc(c & (k0 + 1)) & 1) ? -sg.y : sg.y,
                         (__popc(c & (k0 + 2)) & 1) ? -sg.z : sg.z, (__popc(c & (k0 + 3)) & 1) ? -sg.w : sg.w);
      } else {
        sv = __ldg(reinterpret_cast<const float4*>(S + (size_t)c * D) + (i & 31));
      }
      const float v[4] = {sv.x, sv.y, sv.z, sv.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = f16_bits(v[e]);
        lo[e] = f16_bits(v[e] - __half2float(__float2half_rn(v[e])));
      }
      *reinterpret_cast<uint2*>(Bhi + umma_off(c, k0)) = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
      *reinterpret_cast<uint2*>(Blo + umma_off(c, k0)) = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
    }
    if (warp == 0) {  // max_c ||S_c|| (rounded up)
      float m = 0.f;
      for (int c = lane; c < D; c += 32) {
        float sn;
        if (P.qjl_srht) {
          sn = sqrtf((float)D);
        } else {
          const float4* row = reinterpret_cast<const float4*>(S + (size_t)c * D);
          float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int i = 0; i < D / 4; ++i) {
            const float4 v = __ldg(row + i);
            a4.x = fmaf(v.x, v.x, a4.x);
            a4.y = fmaf(v.y, v.y, a4.y);
            a4.z = fmaf(v.z, v.z, a4.z);
            a4.w = fmaf(v.w, v.w, a4.w);
          }
          sn = sqrtf((a4.x + a4.y) + (a4.z + a4.w));
        }
        m = fmaxf(m, sn * 1.0001f);
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) ts.smax = m;
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B tiles: read by the tensor cores
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const CodeLut lut = code_lut_at(lut_at, lut_j);
  const uint32_t tmem = ts.tmem + (uint32_t)G * 256u;  // group's accumulators: rotation, sketch (+ 128)
  const uint32_t trow = tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(64 * h);
  const float smax = ts.smax;

  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 127) / 128;
  // instruction descriptors: D f32, M = 128, N = 128; A, B bf16 (rotation) or f16 (sketch), K-major
  const uint32_t id_f16 = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
  const uint32_t id_bf16 = id_f16 | (1u << 7) | (1u << 10);
  const float k1 = 6e-5f, k2 = 4e-7f;  // the sketch bound of quantize_keys_tc_kernel
  const int row = 32 * sp + lane;
  uint32_t ph_rot = 0, ph_sk = 0;
  bool failed = false;

  // a warp copies 8 rows x 4 chunks of 16 bytes per step: chunk 4 ci + lane / 8 of row
  // 16 wg + 8 rh + (lane & 7)
  const int lr = 16 * wg + (lane & 7), lc = lane >> 3;
  for (long long tile = (long long)blockIdx.x * 2 + G; tile < n_tiles && !failed; tile += 2LL * gridDim.x) {
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      const long long tk = tile * 128 + lr + 8 * rh;
      const long long n = tk * P.hkv + head;
      const bool rin = tk < n_tok && n < n_vec;
      const __nv_bfloat16* rp = x + (rin ? (size_t)n * P.dh : 0);
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) {
        const int c = 4 * ci + lc;
        const bool in = rin && 8 * c < P.dh;
        cp_async16(buf + umma_off(lr + 8 * rh, 8 * c), in ? rp + 8 * c : x, in ? 16 : 0);
      }
    }
    cp_async_commit();
    cp_async_wait_all();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    bt_bar(G, GT);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (gt == 0) {  // Z = X (H diag(sigma))^T: 8 k-steps
      const uint32_t a = smem_u32(buf), b = smem_u32(Brot);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) bt_mma(tmem, umma_desc(a + 256 * ks), umma_desc(b + 256 * ks), id_bf16, ks > 0);
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(&ts.mbar[G][0])));
    }
    // ---- norm of the row from its bf16 inputs (exact squares, balanced fp32 trees; the two
    // column halves exchange their sums), while the rotation runs
    const long long tok = tile * 128 + row;
    const long long nrow = tok * P.hkv + head;
    const bool ok = tok < n_tok && nrow < n_vec;
    {
      float q2[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(buf + umma_off(row, 64 * h + 8 * c));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
          q2[4 * c + k] = lo * lo + hi * hi;
        }
      }
      ts.part[G][h][row] = tree32(q2);
    }
    if (!bt_wait(&ts.mbar[G][0], ph_rot)) {
      atomicOr(&g_quant_err, TQ_DEVERR_TIMEOUT);
      failed = true;
    }
    ph_rot ^= 1u;
    // the input tile is read (it is overwritten below), the sums are exchanged; one verdict on the wait
    failed = bt_bar_or(G, GT, failed);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const float s2 = ts.part[G][0][row] + ts.part[G][1][row];
    const float nrm = sqrtf(s2);
    const bool zero = nrm < kZeroNorm;
    const float inv = zero ? 0.f : sqrtf(1.0f / s2);  // z = H (sigma x) / n
    if (ok && h == 0 && !failed) norms[nrow] = zero ? 0.f : nrm;

    // ---- codes of 64 coordinates (two words per plane), residual limbs over the input tile
    uint32_t cw[2][4];
    float rsum = 0.f;
#pragma unroll 1
    for (int cc = 0; cc < 2 && !failed; ++cc) {
      uint32_t v[32];
      bt_ld32(trow + (uint32_t)(32 * cc), v);
      uint32_t acc[4] = {0u, 0u, 0u, 0u};
      float sq[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float z = __fmaf_rn(__uint_as_float(v[j]), inv, 0.f);  // +0 for zero rows
        const uint2 rec = code_record(z, lut);
        acc[j >> 3] += rec.y << (j & 7);
        const float r = z - __uint_as_float(rec.x);
        v[j] = __float_as_uint(r);
        sq[j] = r * r;
      }
      planes_of(acc, cw[cc]);
      rsum += tree32(sq);
      // residual limbs: hi over the input tile's first half, lo over the second
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float r0 = __uint_as_float(v[8 * c8 + 2 * e]), r1 = __uint_as_float(v[8 * c8 + 2 * e + 1]);
          hw[e] = pack_f16(r0, r1);
          lw[e] = pack_f16(r0 - f16lo(hw[e]), r1 - f16hi(hw[e]));
        }
        const uint32_t off = umma_off(row, 64 * h + 32 * cc + 8 * c8);
        *reinterpret_cast<uint4*>(buf + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(buf + kBtTile + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    if (ok && !failed) {
      uint32_t* cp = codes + (size_t)nrow * BITS * 4 + 2 * h;
#pragma unroll
      for (int p = 0; p < BITS; ++p) *reinterpret_cast<uint2*>(cp + 4 * p) = make_uint2(cw[0][p], cw[1][p]);
    }

    // ---- S r: 3 limb products x 8 k-steps into the sketch accumulator
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    bt_bar(G, GT);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    ts.part[G][h][row] = rsum;  // every thread of the group has read the norm sums (barrier above)
    if (gt == 0 && !failed) {
      const uint32_t a_hi = smem_u32(buf), a_lo = smem_u32(buf + kBtTile), b_hi = smem_u32(Bhi), b_lo = smem_u32(Blo);
#pragma unroll
      for (int pss = 0; pss < 3; ++pss) {
        if (pss == 2 && P.qjl_srht) break;  // structured S: exact in f16, no lo limb
        const uint32_t a = pss == 1 ? a_lo : a_hi, b = pss == 2 ? b_lo : b_hi;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          bt_mma(tmem + 128, umma_desc(a + 256 * ks), umma_desc(b + 256 * ks), id_f16, (pss > 0 || ks > 0) ? 1u : 0u);
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(&ts.mbar[G][1])));
    }
    if (!failed && !bt_wait(&ts.mbar[G][1], ph_sk)) {
      atomicOr(&g_quant_err, TQ_DEVERR_TIMEOUT);
      failed = true;
    }
    ph_sk ^= 1u;
    failed = bt_bar_or(G, GT, failed);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const float rr = ts.part[G][0][row] + ts.part[G][1][row];  // ||r||^2 in z units
    const float rn = sqrtf(rr);
    const float bmax = fmaf(smax, fmaf(k1, rn, k2), fmaf(k2, rn, k2));
    uint32_t sw[2] = {0u, 0u};
#pragma unroll 1
    for (int cc = 0; cc < 2 && !failed; ++cc) {
      uint32_t v[32];
      bt_ld32(trow + 128u + (uint32_t)(32 * cc), v);
      uint32_t neg = 0, pend = 0;
#pragma unroll
      for (int j = 31; j >= 0; --j) {
        uint32_t lt;
        asm("set.lt.u32.f32 %0, %1, %2;" : "=r"(lt) : "f"(fabsf(__uint_as_float(v[j]))), "f"(bmax));
        asm("shf.l.wrap.b32 %0, %1, %2, 1;" : "=r"(neg) : "r"(v[j]), "r"(neg));
        asm("shf.l.wrap.b32 %0, %1, %2, 1;" : "=r"(pend) : "r"(lt), "r"(pend));
      }
      uint32_t word = ~neg;
      if (zero) {
        word = 0xffffffffu;
        pend = 0u;
      }
      if (!ok) pend = 0u;
      // fp32 recomputation of the uncertain entries from the limbs, one entry per pass of
      // the warp; lane l covers coordinates 4l .. 4l + 3
      while (true) {
        const unsigned ball = __ballot_sync(0xffffffffu, pend != 0u);
        if (ball == 0u) break;
        const int src = __ffs(ball) - 1;
        const int j = __shfl_sync(0xffffffffu, __ffs(pend) - 1, src);
        const int frow = 32 * sp + src, c = 64 * h + 32 * cc + j, k0 = 4 * lane;
        const uint2 ah = *reinterpret_cast<const uint2*>(buf + umma_off(frow, k0));
        const uint2 al = *reinterpret_cast<const uint2*>(buf + kBtTile + umma_off(frow, k0));
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
      sw[cc] = word;
    }
    if (ok && !failed) {
      *reinterpret_cast<uint2*>(signs + (size_t)nrow * 4 + 2 * h) = make_uint2(sw[0], sw[1]);
      if (h == 0) rnorms[nrow] = zero ? 0.f : sqrtf(rr * (1.0f / D));  // exact scaling by a power of two
    }
    // the input / limb buffer, the partial sums and the accumulators are rewritten by the next tile
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    failed = bt_bar_or(G, GT, failed);
  }
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(ts.tmem), "r"(512));
}


// ------------------------------------------------------------------ dense Pi without the sketch
//
// Values, and keys without the QJL sketch, with the dense rotation: the
// rotation Z = X Pi^T runs on tcgen05 against Pi's three bf16 limbs (24
// significant bits, as in quantize_warp_kernel) staged once per CTA as B
// tiles: 24 steps per 128-token tile instead of the 384 mma.sync of the
// warp tiles, which are tensor-bound.  Four groups of 4 warps, one row per
// thread (its 128 rotated coordinates in four tcgen05.ld chunks); the next
// tile is copied as soon as the rotation has read the current one.
constexpr int kBvGroups = 4;

struct BvShared {
  uint64_t mbar[kBvGroups];
  uint32_t tmem;
};

__host__ __device__ constexpr size_t bv_smem_bytes(int J) {
  return 3 * kBtTile + kBvGroups * kBtTile + sizeof(BvShared) + lut_bytes(J, true);
}

// ROLE: 0 values, 2 keys with a scale (EDEN / length-renormalized: rnorms = d / sum z C),
// 3 keys without either.  grid (x, Hkv): CTA (x, h) takes tiles 4 x + G (+ 4 gridDim.x).
template <int BITS, int ROLE>
__global__ void __launch_bounds__(kBtThreads, 1)
    quantize_bv_kernel(const __grid_constant__ KParams P, const __nv_bfloat16* __restrict__ x, long long n_vec,
                       uint32_t* __restrict__ codes, float* __restrict__ norms, float* __restrict__ rnorms,
                       int lut_j) {
  constexpr int NG = kBvGroups, GT = kBtThreads / NG;  // 4 warps per group
  constexpr bool KEY = ROLE != 0;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* Bpi = smem_raw;  // [3 limbs][128 x 128 bf16]
  unsigned char* buf0 = smem_raw + 3 * kBtTile;
  BvShared& ts = *reinterpret_cast<BvShared*>(buf0 + NG * kBtTile);
  unsigned char* lut_at = reinterpret_cast<unsigned char*>(&ts) + sizeof(BvShared);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = warp >> 2, sp = warp & 3, gt = tid % GT;  // group, TMEM sub-partition, thread in group
  const int head = blockIdx.y;
  const float* rot = (KEY ? P.k_rot : P.v_rot) + (size_t)head * D * D;
  unsigned char* buf = buf0 + (size_t)G * kBtTile;

  build_code_lut<BITS, ROLE != 2>(lut_at, lut_j, KEY ? P.kt : P.vt, KEY ? P.kc : P.vc, tid, kBtThreads);
  if (warp == 0) {  // tensor memory: one 128-column rotation accumulator per group
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&ts.tmem)),
                 "r"(512));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int g = 0; g < NG; ++g) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&ts.mbar[g])), "r"(1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // ---- Pi in three bf16 limbs as B tiles: B_l[n][k] = limb l of Pi[n][k]
  for (int i = tid; i < D * (D / 8); i += kBtThreads) {
    const int n = i >> 4, k0 = 8 * (i & 15);
    const float4 a = __ldg(reinterpret_cast<const float4*>(rot + (size_t)n * D + k0));
    const float4 b = __ldg(reinterpret_cast<const float4*>(rot + (size_t)n * D + k0 + 4));
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t l[3][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t h[3][2];
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const float x0 = v[2 * e + f];
        const float l0 = __bfloat162float(__float2bfloat16_rn(x0));
        const float l1 = __bfloat162float(__float2bfloat16_rn(x0 - l0));
        h[0][f] = bf16_bits(x0);
        h[1][f] = bf16_bits(x0 - l0);
        h[2][f] = bf16_bits((x0 - l0) - l1);
      }
#pragma unroll
      for (int t = 0; t < 3; ++t) l[t][e] = h[t][0] | (h[t][1] << 16);
    }
#pragma unroll
    for (int t = 0; t < 3; ++t)
      *reinterpret_cast<uint4*>(Bpi + t * kBtTile + umma_off(n, k0)) = make_uint4(l[t][0], l[t][1], l[t][2], l[t][3]);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B tiles: read by the tensor cores
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const CodeLut lut = code_lut_at(lut_at, lut_j);
  const uint32_t tmem = ts.tmem + (uint32_t)G * 128u;
  const uint32_t trow = tmem + ((uint32_t)(32 * sp) << 16);

  const long long n_tok = (n_vec + P.hkv - 1) / P.hkv;
  const long long n_tiles = (n_tok + 127) / 128;
  const uint32_t id_bf16 = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
  const int row = 32 * sp + lane;
  uint32_t ph = 0;
  bool failed = false;

  // a warp copies 8 rows x 4 chunks of 16 bytes per step: chunk 4 ci + lane / 8 of row
  // 32 sp + 8 rh + (lane & 7)
  const int lr = 32 * sp + (lane & 7), lc = lane >> 3;
  auto load_tile = [&](long long tl) {
#pragma unroll
    for (int rh = 0; rh < 4; ++rh) {
      const long long tk = tl * 128 + lr + 8 * rh;
      const long long n = tk * P.hkv + head;
      const bool rin = tk < n_tok && n < n_vec;
      const __nv_bfloat16* rp = x + (rin ? (size_t)n * P.dh : 0);
#pragma unroll
      for (int ci = 0; ci < 4; ++ci) {
        const int c = 4 * ci + lc;
        const bool in = rin && 8 * c < P.dh;
        cp_async16(buf + umma_off(lr + 8 * rh, 8 * c), in ? rp + 8 * c : x, in ? 16 : 0);
      }
    }
    cp_async_commit();
  };
  const long long tstride = (long long)NG * gridDim.x;
  long long tile = (long long)blockIdx.x * NG + G;
  if (tile < n_tiles) load_tile(tile);
  for (; tile < n_tiles && !failed; tile += tstride) {
    cp_async_wait_all();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    bt_bar(G, GT);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (gt == 0) {  // Z = X Pi^T: 3 limbs x 8 k-steps
      const uint32_t a = smem_u32(buf), b = smem_u32(Bpi);
#pragma unroll
      for (int t = 0; t < 3; ++t)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          bt_mma(tmem, umma_desc(a + 256 * ks), umma_desc(b + (uint32_t)(t * kBtTile) + 256 * ks), id_bf16,
                 (t > 0 || ks > 0) ? 1u : 0u);
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(&ts.mbar[G])));
    }
    // ---- norm of the row from its bf16 inputs (exact squares, balanced fp32 trees), while the rotation runs
    const long long tok = tile * 128 + row;
    const long long nrow = tok * P.hkv + head;
    const bool ok = tok < n_tok && nrow < n_vec;
    float hs[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float q2[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(buf + umma_off(row, 64 * q + 8 * c));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);
          q2[4 * c + k] = lo * lo + hi * hi;
        }
      }
      hs[q] = tree32(q2);
    }
    const float s2 = hs[0] + hs[1];
    if (!bt_wait(&ts.mbar[G], ph)) {
      atomicOr(&g_quant_err, TQ_DEVERR_TIMEOUT);
      failed = true;
    }
    ph ^= 1u;
    failed = bt_bar_or(G, GT, failed);  // the input tile is read; one verdict on the wait
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (tile + tstride < n_tiles && !failed) load_tile(tile + tstride);
    const float nrm = sqrtf(s2);
    const bool zero = nrm < kZeroNorm;
    const float inv = zero ? 0.f : sqrtf((float)D / s2);  // z = sqrt(d) Pi x / n
    if (ok && !failed) norms[nrow] = zero ? 0.f : nrm;

    // ---- codes of the row's 128 coordinates (four words per plane)
    uint32_t cw[4][4];
    float ssum = 0.f;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t v[32];
      if (!failed) bt_ld32(trow + (uint32_t)(32 * cc), v);
      uint32_t acc[4] = {0u, 0u, 0u, 0u};
      float sq[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float z = __fmaf_rn(__uint_as_float(v[j]), inv, 0.f);  // +0 for zero rows
        if constexpr (ROLE == 2) {
          const uint2 rec = code_record(z, lut);
          acc[j >> 3] += rec.y << (j & 7);
          sq[j] = fabsf(z) * fabsf(__uint_as_float(rec.x));  // z C >= 0
        } else {
          acc[j >> 3] += code_spread(z, lut) << (j & 7);
        }
      }
      planes_of(acc, cw[cc]);
      if constexpr (ROLE == 2) ssum += tree32(sq);
    }
    if (ok && !failed) {
      uint32_t* cp = codes + (size_t)nrow * BITS * 4;
#pragma unroll
      for (int p = 0; p < BITS; ++p)
        *reinterpret_cast<uint4*>(cp + 4 * p) = make_uint4(cw[0][p], cw[1][p], cw[2][p], cw[3][p]);
      if constexpr (ROLE == 2) rnorms[nrow] = zero ? 0.f : (float)D / ssum;
    }
    // the accumulator is rewritten by the next tile
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    failed = bt_bar_or(G, GT, failed);
  }
  cp_async_wait_all();  // a prefetch issued before a failed wait
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(ts.tmem), "r"(512));
}

}  // namespace wq
}  // namespace tq
