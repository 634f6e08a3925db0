// Prefill attention over the compressed pages with query tiles (sm_103a).
//
// [Design study] §Transform placement and §Packed format: a prefill chunk's
// queries are scored against the packed pages, not a decoded history;
// [Reconstruction] §6 gives the score of a (query, key) pair, the same as in
// decode.  Every query of a chunk attends to the same compressed pages (each up
// to its own causal position), so a CTA here scores each page for 16 (query,
// head) rows at once instead of one sequence's G heads:
//
//   * the rows are consecutive entries of the chunk's (query, head) list
//     (query i, head h -> entry i G + h), split into units of 16; two
//     mma.m16n8k16 M-tiles of 8 rows each (f16 hi limb in rows 0..7, lo limb
//     in rows 8..15, as in the decode kernel) share every B operand built from
//     the page's bits, so a tile of 8 rows costs the MMAs a decode spends on
//     G <= 8 heads and the operand LOP3s are paid once for both tiles;
//   * the query fragments are those the decode prologue writes for each query
//     as a virtual decode sequence, gathered row by row into the two tiles;
//   * each row carries its own causal bound (the compressed tokens its query
//     sees), its own online-softmax state, and writes the partial of its
//     virtual sequence's head in the decode workspace layout, so the float16
//     window (decode's window split) and the merge (decode's combine kernel)
//     are shared with the virtual-sequence path;
//   * 16 warps: a chunk is 16 pages, warp w scores page w, then owns d / 16
//     value coordinates for all 16 rows; the value planes' Walsh coefficients
//     ride in the weights (one accumulator per tile for both planes).
//
// Compiled for TurboQuant_prod keys (QJL sketch) with 2 or 4 Walsh planes,
// values of 2 bits (+-1 planes) or of 3..4 bits (centroid hi / lo limbs), no
// mixed-channel keys or byte norms: the launcher checks prefill_tiles_ok().
#pragma once

constexpr int kPfThreads = 512;
constexpr int kPfWarps = kPfThreads / 32;  // pages per chunk
constexpr int kPfTiles = 2;                // mma M-tiles per CTA
constexpr int kPfRows = 8 * kPfTiles;      // (query, head) rows per CTA
constexpr int kPfPidCache = 512;           // block-table entries of a split staged in shared memory

struct PfShared {
  uint64_t full[kStages];
  uint4 wf[kPfWarps / 2][kPfTiles][2][2][32];  // weights: [page pair][tile][value plane][k-step][lane]
  float redm[kPfWarps][kPfRows];               // per-warp chunk maxima
  float lsum[kPfWarps][kPfRows];               // per-warp softmax denominators
  float kvsum[kPfWarps][kPfRows];              // per-warp sums of the value operand's constant
  float mfin[kPfRows];
  float kcon[2][kPfRows];  // constant K of the key operand per row: MSE planes, QJL plane
  int vis[kPfRows];        // compressed tokens the row's query sees; -1: no row
  uint32_t vlut[16];
};

// grid (splits, Hkv, batch x units): CTA (s, g, b ups + u) takes rows 16 u .. 16 u + 15 of
// sequence b's (query, head) list against split s of its pages.
template <int D, bool VLUT, int KPF>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tiles_kernel(const __grid_constant__ KParams P, const __grid_constant__ KCache C, int n_query, int ups,
                         float scale, unsigned char* ws, WsLayout L, int max_ctx, int nst) {
  constexpr int E = D / 32, WPL = D / 128, KS = D / 16;
  constexpr int NW = kPfWarps, MT = kPfTiles;
  constexpr int CPW = D / NW;  // value coordinates per warp
  constexpr int CB = CPW / 8;  // n-tiles per warp: 2 at d = 256, 1 at d = 128
  constexpr int NPL = KPF + 1;  // key planes with the sketch's
  constexpr int NPV = VLUT ? 1 : 2;  // weight variants: one per +-1 value plane (its coefficient)
  constexpr int KBITS = KPF == 2 ? 2 : 3;
  static_assert(CB == 1 || CB == 2, "value n-tiles per warp");
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ PfShared sh;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z / ups, u = blockIdx.z % ups;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, t4 = lane & 3;
  const int G = P.G;
  const int st = L.n_comp_splits + 1;
  const int npairs = n_query * G;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float kappa = sqrtf(1.57079632679489662f) / (float)D;
  const int sub = P.sub_bytes;
  const uint32_t xb1 = P.xb1, xb2 = P.xb2;
  const size_t afr_tile = (size_t)NPL * KS * 32;  // uint4 per tile

  // shared memory: query tiles | page stages | page ids of this split
  uint4* afr = reinterpret_cast<uint4*>(dyn);  // [MT][NPL * KS][32]
  unsigned char* stage0 = dyn + (size_t)MT * afr_tile * sizeof(uint4);
  long long* pids = reinterpret_cast<long long*>(stage0 + (size_t)nst * NW * sub);

  // rows: entry 16 u + r of the list is query i = entry / G, head entry % G, virtual sequence
  // b n_query + i; its visible compressed tokens bound the row's scores
  if (tid < kPfRows) {
    const int p = u * kPfRows + tid;
    int vis = -1;
    if (p < npairs) {
      const int v = b * n_query + p / G;
      int T = C.seq_len[v], nc = C.n_compressed[v];
      if (T < 0 || T > max_ctx || nc < 0 || nc > T) {
        atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
        T = min(max(T, 0), max_ctx);
        nc = min(max(nc, 0), T);
      }
      vis = nc;
    }
    sh.vis[tid] = vis;
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
  int ncmax = 0;
#pragma unroll
  for (int r = 0; r < kPfRows; ++r) ncmax = max(ncmax, sh.vis[r]);
  int visr[MT];  // rows g8 and 8 + g8
#pragma unroll
  for (int T = 0; T < MT; ++T) visr[T] = sh.vis[8 * T + g8];
  const int cb = C.parent ? C.parent[(size_t)b * n_query] : b;  // cache row of the chunk's sequence
  int np = (ncmax + kPage - 1) / kPage;
  if (np > C.max_pages) {
    if (tid == 0) atomicOr(&g_decode_err, TQ_DEVERR_SEQ_LEN);
    np = C.max_pages;
  }
  const int p0 = s * L.pages_per_split;
  const int p1 = min(p0 + L.pages_per_split, np);
  const int npg = max(0, p1 - p0);
  const int nchunks = (npg + NW - 1) / NW;
  const int ncache = min(npg, kPfPidCache);
  for (int i = tid; i < ncache; i += kPfThreads) {
    long long pid = C.block_table[(size_t)cb * C.max_pages + p0 + i];
    if (pid < 0 || pid >= C.n_pages) {
      atomicOr(&g_decode_err, TQ_DEVERR_PAGE_INDEX);
      pid = -1;
    }
    pids[i] = pid;
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
  // producer (warp 0, lane i < NW copies page i): chunk k = split pages NW k .. NW k + NW - 1
  // into stage k % nst
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
  // the query fragments come from the prologue (this grid may start while it runs): row r of
  // tile T takes the fragment lanes of its query's head h (rows h and h + 8 of that query's
  // decode tile); rows past the list are zero
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = tid; i < MT * (int)afr_tile; i += kPfThreads) {
    const int ln = i & 31, pk = (i >> 5) % (NPL * KS), T = (i >> 5) / (NPL * KS);
    const int p = u * kPfRows + 8 * T + (ln >> 2);
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (p < npairs) {
      const size_t v = (size_t)b * n_query + p / G;
      const uint4* src = reinterpret_cast<const uint4*>(ws + L.afrag + (v * P.hkv + g) * L.afrag_bytes_per_head);
      val = src[pk * 32 + 4 * (p % G) + (ln & 3)];
    }
    afr[i] = val;
  }
  __syncthreads();
  {
    // K of row `warp` (16 warps, 16 rows): its fragment lanes over all planes and k-blocks;
    // register r of block kk pairs with key bit 2 (kk mod 8) + (r >= 2)
    const int T = warp >> 3, r8 = warp & 7;
    float km = 0.f, kq = 0.f;
    for (int it = lane; it < NPL * KS * 4; it += 32) {
      const int pl = it / (KS * 4), kk = (it / 4) % KS, t4i = it % 4;
      const uint4 a = afr[(size_t)T * afr_tile + (pl * KS + kk) * 32 + r8 * 4 + t4i];
      const uint32_t rr[4] = {a.x, a.y, a.z, a.w};
      float sum = 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float f = xkfac(xpos_key(2 * (kk % 8) + (r >= 2 ? 1 : 0)));
        sum += f * (__half2float(__ushort_as_half((unsigned short)(rr[r] & 0xffffu))) +
                    __half2float(__ushort_as_half((unsigned short)(rr[r] >> 16))));
      }
      if (pl < KPF) km += sum;
      else kq += sum;
    }
    km = warp_sum_f(km);
    kq = warp_sum_f(kq);
    if (lane == 0) {
      sh.kcon[0][warp] = km;
      sh.kcon[1][warp] = kq;
    }
  }

  float accv[MT][CB][4];
#pragma unroll
  for (int T = 0; T < MT; ++T)
#pragma unroll
    for (int c = 0; c < CB; ++c)
#pragma unroll
      for (int r = 0; r < 4; ++r) accv[T][c][r] = 0.f;
  // softmax state of rows g8 and 8 + g8 (identical across warps for m)
  float m_run[MT], l_run[MT], kv_run[MT];
#pragma unroll
  for (int T = 0; T < MT; ++T) {
    m_run[T] = -INFINITY;
    l_run[T] = 0.f;
    kv_run[T] = 0.f;
  }
  // value phase of chunk kc: warp w owns coordinates [w CPW, (w + 1) CPW); runs at the top of
  // iteration kc + 1, overlapping that chunk's key phase
  auto value_phase = [&](int kc) {
    unsigned char* stbase = stage0 + (size_t)(kc % nst) * NW * sub;
#pragma unroll 1
    for (int jg = 0; jg < NW / 2; ++jg) {
      const uint16_t* va = reinterpret_cast<const uint16_t*>(stbase + (size_t)(2 * jg) * sub + P.off_vcodes);
      const uint16_t* vbp = reinterpret_cast<const uint16_t*>(stbase + (size_t)(2 * jg + 1) * sub + P.off_vcodes);
      if (!VLUT) {
        // plane words: page A's 16 slots in bits 0..15, page B's in 16..31; column g8 of n-tile
        // cbk is coordinate warp * CPW + g8 * CB + cbk
        uint32_t u0[CB], u1[CB];
        const int c0 = warp * CPW + g8 * CB;
        if constexpr (CB == 2) {
          const uint32_t a0 = *reinterpret_cast<const uint32_t*>(va + c0), b0 = *reinterpret_cast<const uint32_t*>(vbp + c0);
          const uint32_t a1 = *reinterpret_cast<const uint32_t*>(va + D + c0),
                         b1 = *reinterpret_cast<const uint32_t*>(vbp + D + c0);
          u0[0] = __byte_perm(a0, b0, 0x5410);
          u0[CB - 1] = __byte_perm(a0, b0, 0x7632);
          u1[0] = __byte_perm(a1, b1, 0x5410);
          u1[CB - 1] = __byte_perm(a1, b1, 0x7632);
        } else {
          u0[0] = (uint32_t)va[c0] | ((uint32_t)vbp[c0] << 16);
          u1[0] = (uint32_t)va[D + c0] | ((uint32_t)vbp[D + c0] << 16);
        }
        const int vsh = 12 - 4 * t4;
#pragma unroll
        for (int cbk = 0; cbk < CB; ++cbk) {
          const uint32_t x0 = u0[cbk] << vsh, xm = u1[cbk] << vsh;
#pragma unroll
          for (int ksx = 0; ksx < 2; ++ksx) {
            const int pA = 12 + ksx, pB = 14 + ksx;  // register e = 0, 1
            const uint32_t mA = 0x00010001u << pA, mB = 0x00010001u << pB;
            const uint32_t bA = (x0 & mA) ^ (pA == 14 ? xb2 : xb1), bB = (x0 & mB) ^ (pB == 14 ? xb2 : xb1);
            const uint32_t cA = bA ^ (xm & mA), cB = bB ^ (xm & mB);  // Walsh plane sign ^ magnitude
#pragma unroll
            for (int T = 0; T < MT; ++T) {
              mma16816(accv[T][cbk], sh.wf[jg][T][0][ksx][lane], bA, bB);
              mma16816(accv[T][cbk], sh.wf[jg][T][1][ksx][lane], cA, cB);
            }
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
            // hi halves, then lo halves of the centroid; pair = (token of page A, token of page B)
            const uint32_t h0 = __byte_perm(eA0, eB0, 0x5410), h1 = __byte_perm(eA1, eB1, 0x5410);
            const uint32_t l0 = __byte_perm(eA0, eB0, 0x7632), l1 = __byte_perm(eA1, eB1, 0x7632);
#pragma unroll
            for (int T = 0; T < MT; ++T) {
              const uint4 wfk = sh.wf[jg][T][0][ksx][lane];
              mma16816(accv[T][cbk], wfk, h0, h1);
              mma16816(accv[T][cbk], wfk, l0, l1);
            }
          }
        }
      }
    }
  };
  bool timed_out = false;
  int kstop = nchunks;  // chunks consumed

  for (int k = 0; k <= nchunks; ++k) {
    // softmax of chunk k-1 done (its weights are in sh.wf).  A wait that ran out stops the
    // split here, for every thread alike (no new copies into unfinished phases)
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

    // ---------------- key phase: warp w scores page w of the chunk for both tiles
    const int pi = k * NW + warp;
    const bool pvalid = pi < npg && page_id(pi) >= 0;
    const int pg = p0 + pi;
    const unsigned char* pb = stbase + (size_t)warp * sub;
    float sc[MT][2][2];
    {
      float accm[MT][2][4], accq[MT][2][4];  // [tile][n-tile][frag]
#pragma unroll
      for (int T = 0; T < MT; ++T)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) accm[T][nt][r] = accq[T][nt][r] = 0.f;
      if (pvalid) {
        const uint32_t* kc = reinterpret_cast<const uint32_t*>(pb + P.off_kcodes);
        // raw words of token 2 g8 + nt: word t4 + 4 jw (jw = kk / 8)
        uint32_t rs[2][WPL], rm[KBITS - 1][2][WPL];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int jw = 0; jw < WPL; ++jw) {
            const int tk = 2 * g8 + nt, w = t4 + 4 * jw;
            rs[nt][jw] = kc[tk * E + w];
#pragma unroll
            for (int m = 0; m < KBITS - 1; ++m) rm[m][nt][jw] = kc[((m + 1) * kPage + tk) * E + w];
          }
#pragma unroll
        for (int S = 0; S < KPF; ++S) {
          uint32_t w0[2][WPL], w6[2][WPL], w10[2][WPL];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int jw = 0; jw < WPL; ++jw) {
              uint32_t x = rs[nt][jw];
#pragma unroll
              for (int m = 0; m < KBITS - 1; ++m)
                if (S & (1 << m)) x ^= rm[m][nt][jw];
              w0[nt][jw] = x;
              w6[nt][jw] = x << 6;
              w10[nt][jw] = x << 10;
            }
          const uint4* ap = afr + (size_t)(S * KS) * 32 + lane;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const int jw = kk / 8, i0 = 2 * (kk % 8);
            uint32_t bA[2], bB[2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              bA[nt] = xreg_key(w0[nt][jw], w6[nt][jw], w10[nt][jw], i0, xb1, xb2);
              bB[nt] = xreg_key(w0[nt][jw], w6[nt][jw], w10[nt][jw], i0 + 1, xb1, xb2);
            }
#pragma unroll
            for (int T = 0; T < MT; ++T) {
              const uint4 a = ap[(size_t)T * afr_tile + kk * 32];
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) mma16816(accm[T][nt], a, bA[nt], bB[nt]);
            }
          }
        }
        {
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
          const uint4* ap = afr + (size_t)(KPF * KS) * 32 + lane;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            const int jw = kk / 8, i0 = 2 * (kk % 8);
            uint32_t bA[2], bB[2];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              bA[nt] = xreg_key(q0[nt][jw], q6[nt][jw], q10[nt][jw], i0, xb1, xb2);
              bB[nt] = xreg_key(q0[nt][jw], q6[nt][jw], q10[nt][jw], i0 + 1, xb1, xb2);
            }
#pragma unroll
            for (int T = 0; T < MT; ++T) {
              const uint4 a = ap[(size_t)T * afr_tile + kk * 32];
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) mma16816(accq[T][nt], a, bA[nt], bB[nt]);
            }
          }
        }
      }
      const float* knorm = reinterpret_cast<const float*>(pb + P.off_knorm);
      const float* krn = reinterpret_cast<const float*>(pb + P.off_krnorm);
      float mx[MT];
#pragma unroll
      for (int T = 0; T < MT; ++T) mx[T] = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 4 * t4 + 2 * e + nt;  // column 2 t4 + e of n-tile nt is token 2 (2 t4 + e) + nt
          const int tok = pg * kPage + t;
          const float kn = pvalid ? knorm[t] : 0.f, gm = pvalid ? krn[t] : 0.f;
#pragma unroll
          for (int T = 0; T < MT; ++T) {
            const int rho = 8 * T + g8;
            float l = -INFINITY;
            if (pvalid && tok < visr[T]) {
              // +-1 plane sums from the operand sums: 2 D - K
              const float mse = 2.f * (accm[T][nt][e] + accm[T][nt][e + 2]) - sh.kcon[0][rho];
              const float qj = 2.f * (accq[T][nt][e] + accq[T][nt][e + 2]) - sh.kcon[1][rho];
              l = scale * kn * (mse * inv_sqrt_d + kappa * gm * qj);
            }
            sc[T][nt][e] = l;
            mx[T] = fmaxf(mx[T], l);
          }
        }
      }
#pragma unroll
      for (int T = 0; T < MT; ++T) {
        mx[T] = fmaxf(mx[T], __shfl_xor_sync(0xffffffffu, mx[T], 1));
        mx[T] = fmaxf(mx[T], __shfl_xor_sync(0xffffffffu, mx[T], 2));
        if (t4 == 0) sh.redm[warp][8 * T + g8] = mx[T];
      }
    }
    __syncthreads();
    // ---------------- online softmax: every lane tracks rows g8 and 8 + g8
    {
      const float* vnorm = reinterpret_cast<const float*>(pb + P.off_vnorm);
      float alpha[MT];
      bool rescale = false;
#pragma unroll
      for (int T = 0; T < MT; ++T) {
        const int rho = 8 * T + g8;
        float cm = sh.redm[0][rho];
#pragma unroll
        for (int w = 1; w < NW; ++w) cm = fmaxf(cm, sh.redm[w][rho]);
        const float mnew = fmaxf(m_run[T], cm);
        alpha[T] = 1.f;
        if (mnew != -INFINITY) {
          alpha[T] = expf(m_run[T] - mnew);
          m_run[T] = mnew;
        }
        rescale = rescale || alpha[T] != 1.f;
        // weights of this warp's page in A-fragment order of its page pair: token
        // t = 4 t4 + 2 e + nt -> k-step nt, lane (g8, t4), component 2 e (hi) / 2 e + 1 (lo),
        // half = page parity within the pair; one copy per value plane with its coefficient
        float ls = 0.f, kvs = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int t = 4 * t4 + 2 * e + nt;
            float wgt = 0.f;
            if (sc[T][nt][e] != -INFINITY) {
              const float ex = expf(sc[T][nt][e] - m_run[T]);
              ls += ex;
              wgt = ex * vnorm[t] * inv_sqrt_d;
            }
            const int xp = xpos_val(t);
            if (!VLUT) wgt *= xdelta_inv(xp);  // +-1 value planes read slot t as base + b delta
#pragma unroll
            for (int pv = 0; pv < NPV; ++pv) {
              const float wv = VLUT ? wgt : wgt * P.avw[pv];
              __half hi, lo;
              split_f16(wv, hi, lo);
              if (!VLUT) kvs += (__half2float(hi) + __half2float(lo)) * xkfac(xp);
              uint16_t* dst = reinterpret_cast<uint16_t*>(&sh.wf[warp >> 1][T][pv][0][0]) +
                              ((nt * 32 + lane) * 4 + 2 * e) * 2 + (warp & 1);
              dst[0] = __half_as_ushort(hi);
              dst[2] = __half_as_ushort(lo);
            }
          }
        l_run[T] = l_run[T] * alpha[T] + ls;
        kv_run[T] = kv_run[T] * alpha[T] + kvs;
      }
      if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
        for (int T = 0; T < MT; ++T)
#pragma unroll
          for (int c = 0; c < CB; ++c)
#pragma unroll
            for (int r = 0; r < 4; ++r) accv[T][c][r] *= alpha[T];
      }
    }
  }
  drain_after_timeout(sh.full, timed_out, kstop, nchunks, nst, nst - 2);
  // ---- partials of every row's (virtual sequence, head)
#pragma unroll
  for (int T = 0; T < MT; ++T) {
    float ls = l_run[T], kvl = kv_run[T];
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    kvl += __shfl_xor_sync(0xffffffffu, kvl, 1);
    kvl += __shfl_xor_sync(0xffffffffu, kvl, 2);
    if (t4 == 0) {
      sh.lsum[warp][8 * T + g8] = ls;
      sh.kvsum[warp][8 * T + g8] = kvl;
      if (warp == 0) sh.mfin[8 * T + g8] = m_run[T];
    }
  }
  __syncthreads();
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
#pragma unroll
  for (int T = 0; T < MT; ++T) {
    const int rho = 8 * T + g8, p = u * kPfRows + rho;
    if (p >= npairs) continue;
    const size_t head = ((size_t)b * n_query + p / G) * P.hq + (size_t)g * G + p % G;
    // acc_rot = (hi-limb row + lo-limb row); +-1 value planes: 2 D - K with K summed over every
    // warp's tokens and both planes (the LUT limbs need no correction)
    float kv = 0.f;
    if (!VLUT) {
#pragma unroll
      for (int w = 0; w < NW; ++w) kv += sh.kvsum[w][rho];
    }
    const float pm = VLUT ? 1.f : 2.f;
    // columns 2 t4 and 2 t4 + 1 of n-tile cbk are coordinates warp CPW + (2 t4) CB + cbk and
    // warp CPW + (2 t4 + 1) CB + cbk: 2 CB adjacent coordinates, one vector store
    float o[2 * CB];
#pragma unroll
    for (int cbk = 0; cbk < CB; ++cbk) {
      o[cbk] = pm * (accv[T][cbk][0] + accv[T][cbk][2]) - kv;
      o[CB + cbk] = pm * (accv[T][cbk][1] + accv[T][cbk][3]) - kv;
    }
    vstore_f32<2 * CB>(acc + (head * st + s) * D + warp * CPW + 2 * t4 * CB, o);
  }
  if (tid < kPfRows) {
    const int p = u * kPfRows + tid;
    if (p < npairs) {
      const size_t head = ((size_t)b * n_query + p / G) * P.hq + (size_t)g * G + p % G;
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) l += sh.lsum[w][tid];
      ml[(head * st + s) * 2 + 0] = sh.mfin[tid];
      ml[(head * st + s) * 2 + 1] = l;
    }
  }
}

// The float16 window of every virtual sequence of the chunk (decode's window split), grid
// (Hkv, batch x n_query).
template <int D>
__global__ void __launch_bounds__(kMmaThreads)
    prefill_attn_window_kernel(const __grid_constant__ KParams P, const __grid_constant__ KCache C, const void* q,
                               int dtype, float scale, unsigned char* ws, WsLayout L, int max_ctx) {
  extern __shared__ __align__(128) unsigned char dyn[];
  window_split<D>(P, C, q, dtype, scale, nullptr, ws, L, max_ctx, blockIdx.x, blockIdx.y, dyn);
}
