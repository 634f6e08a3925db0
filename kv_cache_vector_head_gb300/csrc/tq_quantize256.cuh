// Direct-slot quantize of d = 256 keys and values into the paged cache (sm_103a):
// included by tq_quantize.cu after the page-store helpers.
//
// [Reconstruction] §5 Steps 1-5 (norm, rotation, Lloyd-Max code) and §6 (residual,
// gamma, QJL signs of S r); [Design study] §CPU and WASM kernel design ("Append-time key
// kernel"), §Packed format.  Same decisions as quantize_tile, organised for throughput:
//
//   * a CTA of 16 warps owns a tile of 64 tokens of one kv head and loops over tiles
//     (persistent per head); warp w quantizes tokens 4 w .. 4 w + 3 of the tile with the
//     vector in registers (coordinate 32 e + lane in register e): fp32 norm by a balanced
//     tree, the rotation as a shuffle Walsh-Hadamard transform with the sign flips (FWHT
//     kind), codes against the float32 boundaries, sign-magnitude planes by warp ballots;
//   * keys with the Gaussian sketch: S is staged once per CTA in shared memory as f16 in
//     mma.m16n8k16 B-fragment order (128 KB, with its row norms), the residuals of the
//     tile as f16 hi / lo limbs in A-fragment order; S r runs on the tensor cores with
//     both limbs of r against S's hi limb (warp w: rows 16 w .. 16 w + 15 for all 64
//     tokens).  An entry whose magnitude lies within a certified bound of the f16 rounding
//     and accumulation error (1.16 * 2^-11 ||r|| ||S_j|| + 2^-20 (||r|| + ||S_j||)) is recomputed in fp32 by
//     the warp (r from its two limbs, S_j from global memory), so every sign is that of
//     the fp32 product, as in quantize_tile.  The structured sketch takes the signs of a
//     warp transform of sigma_S * r instead;
//   * values (direct256_values_kernel): one warp owns a page group of 16 tokens with lane l
//     holding coordinates 8 l .. 8 l + 7, the coordinate-major 16-slot plane words built in
//     registers and written whole where the group fills a page (prefill), bitwise atomics
//     elsewhere.
// Layers outside this kernel's scope (dense rotation, mixed-channel keys, byte norms, the
// KIVI arm) take append_direct_kernel.

namespace tq {
namespace q256 {

constexpr int D = 256, E = D / 32;
constexpr int NW = 16, NT = 32 * NW;  // warps, threads
constexpr int TILE = 64;              // tokens per tile
constexpr int VPW = TILE / NW;        // tokens per warp in the vector phase
constexpr int MT = TILE / 16;         // m-tiles of the sketch product
constexpr int KS = D / 16;            // k-steps
constexpr int NTL = D / 8;            // n-tiles (rows of S)
constexpr int NTW = NTL / NW;         // n-tiles per warp (2)

struct Tile {
  long long row[TILE];                   // input row of each token
  uint32_t sw[TILE][E];                  // sign words
  float rn[TILE];                        // ||r|| of each token, z units (certification bound)
  long long page[TILE];
  int slot[TILE];
};
constexpr size_t kSBBytes = (size_t)NTL * KS * 32 * sizeof(uint2);        // S, f16 B fragments
constexpr size_t kSABytes = (size_t)MT * KS * 32 * 4 * sizeof(uint32_t);   // one residual limb
__host__ __device__ constexpr size_t smem_bytes(bool sketch) {
  return sizeof(Tile) + (sketch ? kSBBytes + D * sizeof(float) + 2 * kSABytes : 0);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint4& a, const uint2& b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y));
}

// Halfword index of A-fragment element (token row rr of m-tile mt, coordinate k) in a limb array.
// The fragment of lane tl sits in slot tl ^ 4 on odd k-steps: a warp storing coordinates 32 e + lane
// (k-steps 2e and 2e + 1, 512 bytes apart) then writes 32 distinct banks.
__device__ __forceinline__ int a_index(int mt, int rr, int k) {
  const int ks = k >> 4, kk = k & 15;
  const int tl = ((rr & 7) * 4 + ((kk & 7) >> 1)) ^ ((ks & 1) << 2), reg = (rr >> 3) + 2 * (kk >> 3);
  return ((((mt * KS + ks) * 32 + tl) * 4 + reg) << 1) + (kk & 1);
}

// Element offset of (m-tile mt, token row rr, coordinate 32 e + lane) is a_base(mt, rr, lane) + 512 e.
__device__ __forceinline__ int a_base(int mt, int rr, int lane) { return a_index(mt, rr, lane); }

__device__ __forceinline__ float tree8(const float (&v)[E]) {
  return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

// Unnormalised Walsh-Hadamard transform of a warp-held 256-vector (coordinate 32 e + lane in
// v[e], Sylvester order): across lanes a butterfly step is o + s a with s = -1 on the lanes
// whose bit h is set, then the register levels.
__device__ __forceinline__ void wht256(float (&v)[E], int lane) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
    const float sg = (lane & h) ? -1.f : 1.f;
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = fmaf(sg, v[e], __shfl_xor_sync(0xffffffffu, v[e], h));
  }
#pragma unroll
  for (int h = 1; h < E; h <<= 1)
#pragma unroll
    for (int e = 0; e < E; ++e)
      if ((e & h) == 0) {
        const float lo = v[e], hi = v[e + h];
        v[e] = lo + hi;
        v[e + h] = lo - hi;
      }
}

// Keys (KEY is true; values take direct256_values_kernel).  SK: 0 no sketch (MSE-only / scaled keys), 1 Gaussian S on
// the tensor cores, 2 structured S = H diag(sigma_S).  Direct slots as in append_direct_kernel:
// slot_mapping[t] for input token t, or (slot_mapping == NULL) position p of sequence b at
// input row b seq_tok + p, page block_table[b][p / 16], slot p % 16, for t = b n_c + p.
template <bool KEY, int SK>
__global__ void __launch_bounds__(NT, (KEY && SK == 1) ? 1 : 2) direct256_kernel(const __grid_constant__ KParams P,
                                                          const __grid_constant__ KCache C, const void* x, int dtype,
                                                          long long n_tok, const long long* slot_mapping, int seq_tok,
                                                          int n_c, int lut_j) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Tile& tl = *reinterpret_cast<Tile*>(smem_raw);
  uint2* sB = reinterpret_cast<uint2*>(smem_raw + sizeof(Tile));                       // [NTL][KS][32]
  float* sN = reinterpret_cast<float*>(smem_raw + sizeof(Tile) + kSBBytes);            // [D] row norms
  uint16_t* sAh = reinterpret_cast<uint16_t*>(smem_raw + sizeof(Tile) + kSBBytes + D * sizeof(float));
  uint16_t* sAl = reinterpret_cast<uint16_t*>(smem_raw + sizeof(Tile) + kSBBytes + D * sizeof(float) + kSABytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, t4 = lane & 3;
  const int head = blockIdx.y;
  static_assert(KEY, "values take direct256_values_kernel");
  const int bits = P.kb;
  const int half = 1 << (bits - 1);
  const float* ctab = P.kc;
  const float* ttab = P.kt;
  const float* sigma = P.k_rot + (size_t)head * D;
  const float* Sg = P.qjl_s + (size_t)head * (SK == 1 ? D * D : D);
  const int corr = P.kqjl;  // TQ_KEY_*: the scale modes keep s in gamma's slot

  if constexpr (SK == 1) {
    // S of this head: f16 in B-fragment order (n-tile nt = rows 8 nt .., k-step ks), and row norms
    for (int i = tid; i < NTL * KS * 32; i += NT) {
      const int ln = i & 31, ks = (i >> 5) % KS, nt = i / (32 * KS);
      const int j = 8 * nt + (ln >> 2), k0 = 16 * ks + 2 * (ln & 3);
      const float2 p0 = *reinterpret_cast<const float2*>(Sg + (size_t)j * D + k0);
      const float2 p1 = *reinterpret_cast<const float2*>(Sg + (size_t)j * D + k0 + 8);
      const __half2 h0 = __floats2half2_rn(p0.x, p0.y), h1 = __floats2half2_rn(p1.x, p1.y);
      sB[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
    }
    for (int j = warp; j < D; j += NW) {
      float sq[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float v = __ldg(Sg + (size_t)j * D + e * 32 + lane);
        sq[e] = v * v;
      }
      const float s = warp_sum_f(tree8(sq));
      if (lane == 0) sN[j] = sqrtf(s);
    }
  }
  float sig[E];
#pragma unroll
  for (int e = 0; e < E; ++e) sig[e] = __ldg(sigma + e * 32 + lane);
  // codes through the exact cell table (wq::code_record), after the tile's first barrier
  unsigned char* lut_at = smem_raw + smem_bytes(SK == 1);
  wq::build_code_lut_n<false>(lut_at, lut_j, ttab, ctab, bits, tid, NT);
  const wq::CodeLut lut = wq::code_lut_at(lut_at, lut_j);
  float sgs[E];
  if constexpr (SK == 2) {
#pragma unroll
    for (int e = 0; e < E; ++e) sgs[e] = __ldg(Sg + e * 32 + lane);
  }

  const long long n_tiles = (n_tok + TILE - 1) / TILE;
  for (long long tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const long long t0 = tile * TILE;
    // ---- destinations of the tile's tokens
    if (tid < TILE) {
      const long long t = t0 + tid;
      long long pg = -1, row = t;
      int sl = 0;
      if (t < n_tok) {
        long long sm = -1;
        if (slot_mapping) {
          sm = slot_mapping[t];
        } else {
          const long long bq = t / n_c;
          const int pos = (int)(t - bq * n_c);
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
      tl.page[tid] = pg;
      tl.slot[tid] = pg >= 0 ? sl : -1;
      tl.row[tid] = row;
    }
    for (int i = tid; i < TILE * E; i += NT) (&tl.sw[0][0])[i] = 0u;
    __syncthreads();
    long long rows[VPW];
#pragma unroll
    for (int i = 0; i < VPW; ++i) rows[i] = tl.row[VPW * warp + i];

    // ---- vector phase: warp w, tokens VPW w .. VPW w + VPW - 1; bf16 inputs of the next
    // vector are loaded while the current one is quantized
    unsigned short xn[E];
    auto load_raw = [&](int i) {
      const bool ok = tl.page[VPW * warp + i] >= 0;
      const unsigned short* xp = reinterpret_cast<const unsigned short*>(x) + (rows[i] * P.hkv + head) * P.dh;
#pragma unroll
      for (int e = 0; e < E; ++e) xn[e] = (ok && e * 32 + lane < P.dh) ? xp[e * 32 + lane] : (unsigned short)0;
    };
    if (dtype == TQ_BF16) load_raw(0);
#pragma unroll 1
    for (int i = 0; i < VPW; ++i) {
      const int v = VPW * warp + i;
      const long long pg = tl.page[v];
      const int sl = tl.slot[v];
      float xv[E];
      {
        const long long base = (rows[i] * P.hkv + head) * P.dh;
        const bool ok = pg >= 0;
        if (dtype == TQ_BF16) {
#pragma unroll
          for (int e = 0; e < E; ++e) xv[e] = __uint_as_float((uint32_t)xn[e] << 16);  // bf16 -> fp32, exact
          if (i + 1 < VPW) load_raw(i + 1);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e)
            xv[e] = (ok && e * 32 + lane < P.dh) ? load_elem(x, dtype, base + e * 32 + lane) : 0.f;
        }
      }
      float sq[E];
#pragma unroll
      for (int e = 0; e < E; ++e) sq[e] = xv[e] * xv[e];
      const float n = sqrtf(warp_sum_f(tree8(sq)));
      const bool zero = n < kZeroNorm;
      const float inv = zero ? 0.f : 1.0f / n;
      // z = sqrt(d) Pi x / n with Pi = H diag(sigma) / sqrt(d): z = H (sigma x) / n
      float z[E];
#pragma unroll
      for (int e = 0; e < E; ++e) z[e] = xv[e] * sig[e];
      wht256(z, lane);
#pragma unroll
      for (int e = 0; e < E; ++e) z[e] *= inv;
      uint32_t q[E];  // sign-magnitude code, plane p at bit 8 p
      float cz[E];    // its centroid
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint2 rec = wq::code_record(z[e], lut);
        q[e] = rec.y;
        cz[e] = __uint_as_float(rec.x);
      }
      unsigned char* sb = pg >= 0 ? C.pool + ((size_t)pg * P.hkv + head) * (size_t)P.sub_bytes : nullptr;
      // code planes: word e of plane p from one ballot (plane 0: sign side, planes 1..: magnitude bits)
#pragma unroll
      for (int e = 0; e < E; ++e) {
        for (int p = 0; p < bits; ++p) {
          const uint32_t wv = __ballot_sync(0xffffffffu, (q[e] >> (8 * p)) & 1u);
          if (lane == e && sb) reinterpret_cast<uint32_t*>(sb + P.off_kcodes)[(p * kPage + sl) * E + e] = wv;
        }
      }
      if (lane == 0 && sb) reinterpret_cast<float*>(sb + P.off_knorm)[sl] = zero ? 0.f : n;
      if (corr == TQ_KEY_EDEN || corr == TQ_KEY_RENORM) {
        // the unbiased scale s = d / sum_j z_j C[idx_j] (z and its centroid share a sign)
        float tz[E];
#pragma unroll
        for (int e = 0; e < E; ++e) tz[e] = z[e] * cz[e];
        const float a = warp_sum_f(tree8(tz));
        if (lane == 0 && sb) reinterpret_cast<float*>(sb + P.off_krnorm)[sl] = zero ? 0.f : (float)D / a;
      }
      if (corr != TQ_KEY_QJL) continue;
      // residual (z units) and gamma = ||r|| / sqrt(d)
      float r[E], r2[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        r[e] = zero ? 0.f : z[e] - cz[e];
        r2[e] = r[e] * r[e];
      }
      const float rr = sqrtf(warp_sum_f(tree8(r2)));
      if (lane == 0 && sb) reinterpret_cast<float*>(sb + P.off_krnorm)[sl] = zero ? 0.f : rr * 0.0625f;
      if constexpr (SK == 2) {
        // structured sketch: signs of H (sigma_S * r), one word per register
        float a[E];
#pragma unroll
        for (int e = 0; e < E; ++e) a[e] = r[e] * sgs[e];
        wht256(a, lane);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const unsigned w = __ballot_sync(0xffffffffu, (zero || a[e] >= 0.f) ? 1u : 0u);
          if (lane == e) tl.sw[v][e] = w;
        }
      } else if constexpr (SK == 1) {
        if (lane == 0) tl.rn[v] = rr;
        const int ab = a_base(v >> 4, v & 15, lane);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const __half h = __float2half_rn(r[e]);
          const __half lo = __float2half_rn(r[e] - __half2float(h));
          sAh[ab + 512 * e] = __half_as_ushort(h);
          sAl[ab + 512 * e] = __half_as_ushort(lo);
        }
      }
    }
    __syncthreads();

    if constexpr (KEY && SK == 1) {
      if (corr == TQ_KEY_QJL) {
        // ---- sketch phase: warp w, rows 16 w .. 16 w + 15 of S r for all 64 tokens
        float acc[MT][NTW][4];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int q = 0; q < NTW; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[m][q][c] = 0.f;
        // both limbs of r against S's hi limb: the products are exact, so the error left is S's
        // own rounding (2^-11 relative), the 32 chained fp32 accumulations and subnormal limbs
        const uint4* A4 = reinterpret_cast<const uint4*>(sAh);
        const uint4* A4l = reinterpret_cast<const uint4*>(sAl);
#pragma unroll 2
        for (int ks = 0; ks < KS; ++ks) {
          uint2 b[NTW];
#pragma unroll
          for (int q = 0; q < NTW; ++q) b[q] = sB[((NTW * warp + q) * KS + ks) * 32 + lane];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            const uint4 a = A4[(m * KS + ks) * 32 + (lane ^ ((ks & 1) << 2))];  // slot swizzle of a_index
            const uint4 al = A4l[(m * KS + ks) * 32 + (lane ^ ((ks & 1) << 2))];
#pragma unroll
            for (int q = 0; q < NTW; ++q) {
              mma_f16(acc[m][q], a, b[q]);
              mma_f16(acc[m][q], al, b[q]);
            }
          }
        }
        // signs; entries within the certified bound are recomputed in fp32 by the whole warp
        uint32_t sbits = 0, unc = 0;  // bit (m NTW + q) 4 + c
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int q = 0; q < NTW; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int v = 16 * m + g8 + 8 * (c >> 1);
              const int j = 8 * (NTW * warp + q) + 2 * t4 + (c & 1);
              const float rnv = tl.rn[v], snj = sN[j];
              // 2^-11 (S's hi limb) + 32 * 17 * 2^-23 (chained accumulation, each step truncating
              // every addend by an ulp) < 1.16 * 2^-11, relative to ||r|| ||S_j||
              const float bound = 1.16f * 0x1p-11f * rnv * snj + 0x1p-20f * (rnv + snj);
              const int bit = (m * NTW + q) * 4 + c;
              if (acc[m][q][c] >= 0.f) sbits |= 1u << bit;
              if (fabsf(acc[m][q][c]) <= bound) unc |= 1u << bit;
            }
        // the uncertain entries two at a time (lane l's lowest pending bit; both rows of S are
        // loaded before either dot product is reduced), no pass where the warp has none
        while (true) {
          int l[2], bit[2];
          bool have[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const unsigned who = __ballot_sync(0xffffffffu, unc != 0u);
            have[u] = who != 0u;
            l[u] = have[u] ? __ffs(who) - 1 : 0;
            bit[u] = __shfl_sync(0xffffffffu, __ffs(unc) - 1, l[u]);
            if (have[u] && lane == l[u]) unc &= unc - 1u;
          }
          if (!have[0]) break;
          float prod[2][E];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int b = have[u] ? bit[u] : bit[0], ll = have[u] ? l[u] : l[0];
            const int c = b & 3, q = (b >> 2) % NTW, m = b / (4 * NTW);
            const int v = 16 * m + (ll >> 2) + 8 * (c >> 1);
            const int j = 8 * (NTW * warp + q) + 2 * (ll & 3) + (c & 1);
            const int ab = a_base(v >> 4, v & 15, lane);
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const int ai = ab + 512 * e;
              const float rv = __half2float(__ushort_as_half(sAh[ai])) + __half2float(__ushort_as_half(sAl[ai]));
              prod[u][e] = rv * __ldg(Sg + (size_t)j * D + e * 32 + lane);
            }
          }
          float dot[2] = {tree8(prod[0]), tree8(prod[1])};
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int u = 0; u < 2; ++u) dot[u] += __shfl_xor_sync(0xffffffffu, dot[u], o);
#pragma unroll
          for (int u = 0; u < 2; ++u)
            if (have[u] && lane == l[u]) sbits = (sbits & ~(1u << bit[u])) | ((dot[u] >= 0.f ? 1u : 0u) << bit[u]);
        }
        // sign words: token v, rows 16 w .. 16 w + 15 are bits 16 (w & 1) .. of word w / 2
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int hv = 0; hv < 2; ++hv) {
            uint32_t part = 0;
#pragma unroll
            for (int q = 0; q < NTW; ++q)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int bit = (m * NTW + q) * 4 + 2 * hv + e;
                part |= ((sbits >> bit) & 1u) << (8 * q + 2 * t4 + e);
              }
            part |= __shfl_xor_sync(0xffffffffu, part, 1);
            part |= __shfl_xor_sync(0xffffffffu, part, 2);
            if (t4 == 0) atomicOr(&tl.sw[16 * m + g8 + 8 * hv][warp >> 1], part << (16 * (warp & 1)));
          }
      }
      __syncthreads();
    }
    if (corr == TQ_KEY_QJL && SK != 0) {
      for (int i = tid; i < TILE * E; i += NT) {
        const int v = i / E, e = i % E;
        if (tl.page[v] >= 0)
          reinterpret_cast<uint32_t*>(C.pool + ((size_t)tl.page[v] * P.hkv + head) * (size_t)P.sub_bytes +
                                      P.off_ksigns)[tl.slot[v] * E + e] = tl.sw[v][e];
      }
    }
    __syncthreads();
  }
  (void)half;
}

// ------------------------------------------------------------------ values, a page group per warp

// Values at d = 256 (FWHT kind): one warp owns a group of 16 tokens, a page's worth.  Lane l holds
// coordinates 8 l .. 8 l + 7 (a bf16 row is one 16-byte load a lane), so the Walsh-Hadamard
// transform takes the three low index levels in registers and the five high ones across lanes,
// and the group's coordinate-major 16-slot plane words build up in the lane's registers: byte p
// of accA[e] / accB[e] holds plane p of coordinate 8 l + e for tokens 0..7 / 8..15.  A group that
// fills one page in slot order leaves as one 16-byte store a lane and plane (and the 16 norms in
// one store); any other group writes each token's bits with bitwise atomics.  Groups: page pp of
// sequence b (slot_mapping == NULL: position p of sequence b at input row b seq_tok + p, page
// block_table[b][p / 16], slot p % 16), or 16 consecutive input tokens (slot_mapping[t]).
constexpr int VNW = 8;  // warps a CTA
__global__ void __launch_bounds__(32 * VNW) direct256_values_kernel(const __grid_constant__ KParams P,
                                                                   const __grid_constant__ KCache C, const void* x,
                                                                   int dtype, long long n_tok,
                                                                   const long long* slot_mapping, int seq_tok,
                                                                   int n_c, int lut_j) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int head = blockIdx.y;
  const int bits = P.vb;
  wq::build_code_lut_n<true>(smem_raw, lut_j, P.vt, P.vc, bits, tid, 32 * VNW);
  const wq::CodeLut lut = wq::code_lut_at(smem_raw, lut_j);
  uint32_t sgm[8];  // sign bit of sigma_j (+-1) for the lane's coordinates 8 lane + e
  {
    const uint4* sp = reinterpret_cast<const uint4*>(P.v_rot + (size_t)head * D) + 2 * lane;
    const uint4 a = __ldg(sp), b = __ldg(sp + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) sgm[e] = w[e] & 0x80000000u;
  }
  __syncthreads();
  const bool vec = dtype == TQ_BF16 && P.dh == D;  // rows of 512 bytes, 16-byte aligned (checked on the host)
  const uint4* xq = reinterpret_cast<const uint4*>(x);
  const long long npp = slot_mapping ? 1 : (n_c + kPage - 1) / kPage;  // pages a sequence
  const long long n_groups = slot_mapping ? (n_tok + 15) / 16 : (n_c > 0 ? n_tok / n_c : 0) * npp;

  // destination and input row of token i = lane (< 16) of group gi
  struct Dst {
    long long pg, off;  // page (-1: none), element offset of the input row
    int sl;
  };
  auto dest = [&](long long gi) -> Dst {
    long long pg = -1, row = 0;
    int sl = -1;
    if (lane < 16 && gi < n_groups) {
      if (slot_mapping) {
        const long long t = gi * 16 + lane;
        if (t < n_tok) {
          row = t;
          const long long sm = slot_mapping[t];  // negative: skipped
          if (sm >= 0) {
            pg = sm / kPage;
            sl = (int)(sm % kPage);
            if (pg >= C.n_pages) {
              atomicOr(&g_quant_err, TQ_DEVERR_SLOT);
              pg = -1;
            }
          }
        }
      } else {
        const long long bq = gi / npp;
        const int pp = (int)(gi - bq * npp), pos = pp * kPage + lane;
        if (pos < n_c) {
          row = bq * seq_tok + pos;
          if (pp < C.max_pages) {
            const long long pid = C.block_table[(size_t)bq * C.max_pages + pp];
            if (pid >= 0 && pid < C.n_pages) {
              pg = pid;
              sl = lane;
            } else {
              atomicOr(&g_quant_err, TQ_DEVERR_SLOT);
            }
          } else {
            atomicOr(&g_quant_err, TQ_DEVERR_SEQ_LEN);
          }
        }
      }
    }
    return Dst{pg, (row * P.hkv + head) * (long long)P.dh, sl};
  };
  auto load = [&](const Dst& d, int i) -> uint4 {  // row of token i of d's group (zeros if it has none)
    const long long oi = __shfl_sync(0xffffffffu, d.off, i);
    const long long pgi = __shfl_sync(0xffffffffu, d.pg, i);
    return (vec && pgi >= 0) ? __ldg(xq + oi / 8 + lane) : make_uint4(0u, 0u, 0u, 0u);
  };
  const long long gstride = (long long)gridDim.x * VNW;
  long long gi = (long long)blockIdx.x * VNW + warp;
  Dst cur = dest(gi);
  // two tokens a pass; the rows of the next two passes (past the group's end: the next group's
  // first ones) are in flight meanwhile, and the next group's destinations are read at its start
  uint4 r0 = load(cur, 0), r1 = load(cur, 1), r2 = load(cur, 2), r3 = load(cur, 3);
  for (; gi < n_groups; gi += gstride) {
    const Dst nxt = dest(gi + gstride);
    const long long pg = cur.pg, off = cur.off;
    const int sl = cur.sl;
    const unsigned vmask = __ballot_sync(0xffffffffu, lane < 16 && pg >= 0);
    const long long pg0 = __shfl_sync(0xffffffffu, pg, 0);
    const bool full = vmask == 0xFFFFu && __all_sync(0xffffffffu, lane >= 16 || (pg == pg0 && sl == lane));
    uint32_t accA[8], accB[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) accA[e] = accB[e] = 0u;
    float nrm = 0.f;  // lane i < 16: the norm of token i
    auto token = [&](int i, const uint4 raw) {
      if (!((vmask >> i) & 1u)) return;  // warp-uniform
      // sigma x (sigma = +-1): bf16 rows exactly, the sign flip as an XOR of the sign bit
      float z[8];
      if (vec) {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          z[2 * k] = __uint_as_float((w[k] << 16) ^ sgm[2 * k]);
          z[2 * k + 1] = __uint_as_float((w[k] & 0xFFFF0000u) ^ sgm[2 * k + 1]);
        }
      } else {
        const long long oi = __shfl_sync(0xffffffffu, off, i);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          z[e] = __uint_as_float(__float_as_uint(8 * lane + e < P.dh ? load_elem(x, dtype, oi + 8 * lane + e) : 0.f) ^
                                 sgm[e]);
      }
      float sq[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) sq[e] = z[e] * z[e];
      const float ss = warp_sum_f(tree8(sq));
      const float n = sqrtf(ss);
      const bool zero = n < kZeroNorm;
      // 1 / n within two ulp (the codes compare z to the boundaries; their exemption band is far wider)
      const float inv = zero ? 0.f : rsqrtf(ss);
      // z = sqrt(d) Pi x / n with Pi = H diag(sigma) / sqrt(d): z = H (sigma x) / n; index bits 3..7
      // (the lane's) across lanes, bits 0..2 (the register's) in registers
#pragma unroll
      for (int h = 1; h < 32; h <<= 1) {
        const float sg = (lane & h) ? -1.f : 1.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) z[e] = fmaf(sg, z[e], __shfl_xor_sync(0xffffffffu, z[e], h));
      }
#pragma unroll
      for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if ((e & h) == 0) {
            const float lo = z[e], hi = z[e + h];
            z[e] = lo + hi;
            z[e + h] = lo - hi;
          }
      uint32_t q[8];  // spread code: plane p at bit 8 p
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = wq::code_spread(z[e] * inv, lut);
      if (lane == i) nrm = zero ? 0.f : n;
      if (full) {
        const int shv = i & 7;
        if (i < 8) {
#pragma unroll
          for (int e = 0; e < 8; ++e) accA[e] |= q[e] << shv;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) accB[e] |= q[e] << shv;
        }
        return;
      }
      // a group that is not one whole page: this token's bits (slot sli of page pgi), coordinate
      // pairs 8 lane + 2 k, + 1 in one 32-bit word
      const long long pgi = __shfl_sync(0xffffffffu, pg, i);
      const int sli = __shfl_sync(0xffffffffu, sl, i);
      unsigned char* sb = C.pool + ((size_t)pgi * P.hkv + head) * (size_t)P.sub_bytes;
      unsigned int* w32 = reinterpret_cast<unsigned int*>(sb + P.off_vcodes) + 4 * lane;
      const unsigned clear = ~((1u << sli) | (1u << (16 + sli)));
      for (int p = 0; p < bits; ++p) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const unsigned b2 = (((q[2 * k] >> (8 * p)) & 1u) << sli) | (((q[2 * k + 1] >> (8 * p)) & 1u) << (16 + sli));
          atomicAnd(w32 + p * (D / 2) + k, clear);
          atomicOr(w32 + p * (D / 2) + k, b2);
        }
      }
      if (lane == 0) reinterpret_cast<float*>(sb + P.off_vnorm)[sli] = zero ? 0.f : n;
    };
#pragma unroll 1
    for (int i = 0; i < 16; i += 2) {
      const uint4 c0 = r0, c1 = r1;
      r0 = r2;
      r1 = r3;
      const Dst& d = i + 4 < 16 ? cur : nxt;
      const int i4 = (i + 4) & 15;
      r2 = load(d, i4);
      r3 = load(d, i4 + 1);
      token(i, c0);
      token(i + 1, c1);
    }
    if (full) {
      unsigned char* sb = C.pool + ((size_t)pg0 * P.hkv + head) * (size_t)P.sub_bytes;
      uint4* dst = reinterpret_cast<uint4*>(sb + P.off_vcodes) + lane;  // coordinates 8 lane .. 8 lane + 7
      for (int p = 0; p < bits; ++p) {
        const uint32_t sel = (uint32_t)p | ((uint32_t)(p + 4) << 4);  // byte p of each operand
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t xa = __byte_perm(accA[2 * k], accA[2 * k + 1], sel);
          const uint32_t xb = __byte_perm(accB[2 * k], accB[2 * k + 1], sel);
          w[k] = __byte_perm(xa, xb, 0x5140);  // word 2k: tokens 0..7 | 8..15 << 8; word 2k + 1 above
        }
        dst[p * (D / 8)] = make_uint4(w[0], w[1], w[2], w[3]);  // plane p: D halfwords, 32 uint4
      }
      if (lane < 16) reinterpret_cast<float*>(sb + P.off_vnorm)[lane] = nrm;
    }
    cur = nxt;
  }
}

}  // namespace q256
}  // namespace tq
