// KIVI-like control arm: decode over its pages on the tensor cores (sm_103a).
//
// [Design study] §Candidate key and value algorithms, arm 3.  A key's channel
// j dequantizes to zk_j + sk_j c_j (float16 scale and zero of the channel in
// the page), a value of token t to zv_t + sv_t c_t.  The two contractions
//   score_h(t) = sum_j q_hj sk_j c_tj + sum_j q_hj zk_j,
//   acc_h(j)   = sum_t (p_ht sv_t) c_tj + sum_t p_ht zv_t
// run on mma.m16n8k16 with operands exact in f16: the b-bit code is split
// into its bits, c = sum_p 2^p bit_p, and each bit plane enters as the f16
// value 2^p sk_j (keys) or 2^p (values) where the bit is set and 0 where it is
// not (one rotate puts the bit at a byte's top, one byte permute spreads it
// over a 16-bit mask, one AND takes the value), so the per-page channel scale
// rides on the code side and the query operand (f16 hi / lo limbs in rows h
// and h + 8, as in the TurboQuant decode) stays fixed for the whole call.  The
// zero terms are plain sums: sum_j q_hj zk_j per page on CUDA cores, and
// sum_t p_ht zv_t with the softmax weights.
//
// Key k-step kk covers 16 channels; the two halves of an f16x2 operand register
// are channels 16 bits apart in the packed token word (channel j and j + 8 at
// 2 bits, j and j + 4 at 4 bits), so that one rotate serves both:
//   KB = 2: b0 = channels (16 kk + t4, 16 kk + t4 + 8), b1 = (16 kk + t4 + 4, 16 kk + t4 + 12)
//   KB = 4: b0 = (16 kk + t4, 16 kk + t4 + 4), b1 = (16 kk + 8 + t4, 16 kk + 12 + t4)
// and the query fragment's columns 2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9 carry those channels.
// Value tiles follow the decode's token order (slot 4 t4 + 2 e + k of pages A, B of a pair).
#pragma once

template <int KB>
__device__ __forceinline__ void kivi_key_channels(int kk, int t4, int (&c)[4]) {
  if (KB == 2) {
    c[0] = 16 * kk + t4;
    c[1] = 16 * kk + t4 + 8;
    c[2] = 16 * kk + t4 + 4;
    c[3] = 16 * kk + t4 + 12;
  } else {
    c[0] = 16 * kk + t4;
    c[1] = 16 * kk + t4 + 4;
    c[2] = 16 * kk + 8 + t4;
    c[3] = 16 * kk + 12 + t4;
  }
}

// 0xFFFF in the low half where bit `pos` of w is set, 0xFFFF in the high half where bit pos + 16
// is: rotate bit pos to bit 7 (pos + 16 lands on bit 23), then replicate the top bits of bytes 0
// and 2.
__device__ __forceinline__ uint32_t kivi_mask(uint32_t w, int pos) {
  uint32_t x, m;
  asm("shf.l.wrap.b32 %0, %1, %1, %2;" : "=r"(x) : "r"(w), "r"((7 - pos) & 31));
  asm("prmt.b32 %0, %1, 0, 0xAA88;" : "=r"(m) : "r"(x));
  return m;
}
// Low half from bit `pos` of wa, high half from bit `pos` of wb.
__device__ __forceinline__ uint32_t kivi_mask2(uint32_t wa, uint32_t wb, int pos) {
  uint32_t xa, xb, m;
  asm("shf.l.wrap.b32 %0, %1, %1, %2;" : "=r"(xa) : "r"(wa), "r"((7 - pos) & 31));
  asm("shf.l.wrap.b32 %0, %1, %1, %2;" : "=r"(xb) : "r"(wb), "r"((7 - pos) & 31));
  asm("prmt.b32 %0, %1, %2, 0xCC88;" : "=r"(m) : "r"(xa), "r"(xb));
  return m;
}

struct KvmShared {
  uint64_t full[kStages];
  uint4 wf[2][kMmaPages / 2][2][32];  // softmax weights x value scale, A-fragment order (chunk parity)
  float redm[kMmaPages][TQ_MAX_GQA];
  float lsum[kMmaPages][TQ_MAX_GQA];
  float zsum[kMmaPages][TQ_MAX_GQA];  // sum_t p_t zv_t
  float mfin[TQ_MAX_GQA];
};

template <int D, int KB, int VB>
__global__ void __launch_bounds__(kMmaThreads, 2) kivi_mma_kernel(const __grid_constant__ KParams P,
                                                                   const __grid_constant__ KCache C, const void* q,
                                                                   int dtype, float scale, float* scores,
                                                                   unsigned char* ws, WsLayout L, int max_ctx,
                                                                   int nst) {
  constexpr int NW = kMmaThreads / 32;  // pages per chunk
  constexpr int KS = D / 16;
  constexpr int KW = D * KB / 32, VW = D * VB / 32;  // code words per token
  constexpr int CPW = D / NW;                        // value coordinates per warp
  constexpr int CB = CPW / 8;
  constexpr int E = D / 32;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ KvmShared sh;
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  if (s == L.n_comp_splits) {  // the float16 window runs as the last split
    window_split<D>(P, C, q, dtype, scale, scores, ws, L, max_ctx, g, b, dyn);
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, t4 = lane & 3;
  const int G = P.G;
  const int st = L.n_comp_splits + 1;
  const size_t head0 = (size_t)b * P.hq + (size_t)g * G;
  const int sub = P.sub_bytes;

  // shared memory: query fragments | query rows (float) | page stages | page ids of this split
  uint4* afr = reinterpret_cast<uint4*>(dyn);                                   // [KS][32]
  float* qs = reinterpret_cast<float*>(dyn + (size_t)KS * 32 * sizeof(uint4));  // [8][D]
  unsigned char* stage0 = reinterpret_cast<unsigned char*>(qs + TQ_MAX_GQA * D);  // [nst][NW][sub]
  long long* pids = reinterpret_cast<long long*>(stage0 + (size_t)nst * NW * sub);

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
  for (int i = tid; i < TQ_MAX_GQA * D; i += kMmaThreads) {
    const int h = i / D, j = i % D;
    qs[i] = (h < G && j < P.dh) ? load_elem(q, dtype, (long long)((head0 + h) * P.dh + j)) : 0.f;  // zero-padded
  }
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&sh.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // query fragments: k-step kk, lane (g8, t4): rows g8 (hi limb) and g8 + 8 (lo limb) of head g8
  // at the channels of this lane's key operand registers
  for (int i = tid; i < KS * 32; i += kMmaThreads) {
    const int kk = i >> 5, ln = i & 31, h = ln >> 2, tt = ln & 3;
    int c[4];
    kivi_key_channels<KB>(kk, tt, c);
    __half hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) split_f16(qs[h * D + c[e]], hi[e], lo[e]);  // rows h >= G are zero
    afr[i] = make_uint4(pack_h2(hi[0], hi[1]), pack_h2(lo[0], lo[1]), pack_h2(hi[2], hi[3]), pack_h2(lo[2], lo[3]));
  }
  __syncthreads();

  auto page_id = [&](int i) -> long long {
    if (i >= npg) return -1;
    if (i < ncache) return pids[i];
    long long pid = C.block_table[(size_t)cb * C.max_pages + p0 + i];
    if (pid < 0 || pid >= C.n_pages) {
      atomicOr(&g_decode_err, TQ_DEVERR_PAGE_INDEX);
      pid = -1;
    }
    return pid;
  };
  auto issue = [&](int k) {  // warp 0: chunk k into stage k % nst, lane i < NW copies page i
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

  float accv[CB][4];
#pragma unroll
  for (int c = 0; c < CB; ++c)
#pragma unroll
    for (int r = 0; r < 4; ++r) accv[c][r] = 0.f;
  float m_run = -INFINITY, l_run = 0.f, z_run = 0.f;  // softmax state of head g8

  // value phase of chunk kc: warp w owns coordinates [w CPW, (w + 1) CPW), column g8 of n-tile
  // cbk is coordinate w CPW + g8 CB + cbk
  auto value_phase = [&](int kc) {
    unsigned char* stbase = stage0 + (size_t)(kc % nst) * NW * sub;
    const uint4(&wfb)[kMmaPages / 2][2][32] = sh.wf[kc & 1];
#pragma unroll 1
    for (int jg = 0; jg < NW / 2; ++jg) {
      const uint32_t* va = reinterpret_cast<const uint32_t*>(stbase + (size_t)(2 * jg) * sub + P.off_vcodes);
      const uint32_t* vbp = reinterpret_cast<const uint32_t*>(stbase + (size_t)(2 * jg + 1) * sub + P.off_vcodes);
      const uint4 wf0 = wfb[jg][0][lane], wf1 = wfb[jg][1][lane];
#pragma unroll
      for (int cbk = 0; cbk < CB; ++cbk) {
        const int c = warp * CPW + g8 * CB + cbk;
        const int wi = (c * VB) >> 5, bit0 = (c * VB) & 31;
#pragma unroll
        for (int ksx = 0; ksx < 2; ++ksx) {
          // slots 4 t4 + ksx (register e = 0) and 4 t4 + 2 + ksx (e = 1) of pages A and B
          const int t0 = 4 * t4 + ksx, t1 = t0 + 2;
          const uint32_t a0 = va[t0 * VW + wi], b0w = vbp[t0 * VW + wi];
          const uint32_t a1 = va[t1 * VW + wi], b1w = vbp[t1 * VW + wi];
          const uint4 wfk = ksx ? wf1 : wf0;
#pragma unroll
          for (int p = 0; p < VB; ++p) {
            const uint32_t two_p = p == 0 ? 0x3C003C00u : p == 1 ? 0x40004000u : p == 2 ? 0x44004400u : 0x48004800u;
            mma16816(accv[cbk], wfk, kivi_mask2(a0, b0w, bit0 + p) & two_p, kivi_mask2(a1, b1w, bit0 + p) & two_p);
          }
        }
      }
    }
  };
  bool timed_out = false;
  int kstop = nchunks;

  for (int k = 0; k <= nchunks; ++k) {
    if (__syncthreads_or(timed_out)) {
      kstop = k;
      break;
    }
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
      float acc[2][2][4];  // [kk parity][n-tile][frag]
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[x][nt][r] = 0.f;
      float zk = 0.f;  // sum_j q_(g8) j zk_j of this page
      if (pvalid) {
        const uint32_t* kc = reinterpret_cast<const uint32_t*>(pb + P.off_kcodes);
        const __half* ksc = reinterpret_cast<const __half*>(pb + P.off_kscale);
        const __half* kzr = reinterpret_cast<const __half*>(pb + P.off_kzero);
#pragma unroll 4
        for (int kk = 0; kk < KS; ++kk) {
          int c[4];
          kivi_key_channels<KB>(kk, t4, c);
          // channel-scale pairs of the two registers, times 2^p for bit plane p (exact in f16)
          __half2 s0 = __halves2half2(ksc[c[0]], ksc[c[1]]), s1 = __halves2half2(ksc[c[2]], ksc[c[3]]);
          const int wb0 = KB == 2 ? kk : 2 * kk, wb1 = KB == 2 ? kk : 2 * kk + 1;
          const int pos0 = ((c[0] * KB) & 31), pos1 = ((c[2] * KB) & 31);
          uint32_t w0[2], w1[2];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int tk = 2 * g8 + nt;  // column g8 of n-tile nt
            w0[nt] = kc[tk * KW + wb0];
            w1[nt] = kc[tk * KW + wb1];
          }
          const uint4 a = afr[kk * 32 + lane];
#pragma unroll
          for (int p = 0; p < KB; ++p) {
            const uint32_t u0 = *reinterpret_cast<const uint32_t*>(&s0), u1 = *reinterpret_cast<const uint32_t*>(&s1);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
              mma16816(acc[kk & 1][nt], a, kivi_mask(w0[nt], pos0 + p) & u0, kivi_mask(w1[nt], pos1 + p) & u1);
            s0 = __hadd2(s0, s0);
            s1 = __hadd2(s1, s1);
          }
        }
        // the zero term on CUDA cores: lane l takes channels l, l + 32, ... for every head
        float zp[TQ_MAX_GQA];
#pragma unroll
        for (int h = 0; h < TQ_MAX_GQA; ++h) zp[h] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float z = __half2float(kzr[e * 32 + lane]);
#pragma unroll
          for (int h = 0; h < TQ_MAX_GQA; ++h)
            if (h < G) zp[h] = fmaf(qs[h * D + e * 32 + lane], z, zp[h]);
        }
#pragma unroll
        for (int h = 0; h < TQ_MAX_GQA; ++h) {
          if (h < G) {
            const float v = warp_sum_f(zp[h]);
            if (g8 == h) zk = v;
          }
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 4 * t4 + 2 * e + nt;  // column 2 t4 + e of n-tile nt is token 2 (2 t4 + e) + nt
          const int tok = pg * kPage + t;
          const bool live = pvalid && g8 < G && tok < nc;
          float l = -INFINITY;
          if (live) {
            l = scale * ((acc[0][nt][e] + acc[0][nt][e + 2]) + (acc[1][nt][e] + acc[1][nt][e + 2]) + zk);
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
    {
      float cm = sh.redm[0][g8];
#pragma unroll
      for (int w = 1; w < NW; ++w) cm = fmaxf(cm, sh.redm[w][g8]);
      float alpha = 1.f;
      const float mnew = fmaxf(m_run, cm);
      if (mnew != -INFINITY) {
        alpha = expf(m_run - mnew);
        m_run = mnew;
      }
      const __half* vsc = reinterpret_cast<const __half*>(pb + P.off_vscale);
      const __half* vzr = reinterpret_cast<const __half*>(pb + P.off_vzero);
      uint16_t* wfh = reinterpret_cast<uint16_t*>(&sh.wf[k & 1][warp >> 1][0][0]);
      float ls = 0.f, zs = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 4 * t4 + 2 * e + nt;
          float wgt = 0.f;
          if (sc[nt][e] != -INFINITY) {
            const float ex = expf(sc[nt][e] - m_run);
            ls += ex;
            wgt = ex * __half2float(vsc[t]);
            zs = fmaf(ex, __half2float(vzr[t]), zs);
          }
          __half hi, lo;
          split_f16(wgt, hi, lo);
          uint16_t* dst = wfh + ((nt * 32 + lane) * 4 + 2 * e) * 2 + (warp & 1);
          dst[0] = __half_as_ushort(hi);
          dst[2] = __half_as_ushort(lo);
        }
      l_run = l_run * alpha + ls;
      z_run = z_run * alpha + zs;
      if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < CB; ++c)
#pragma unroll
          for (int r = 0; r < 4; ++r) accv[c][r] *= alpha;
      }
    }
  }
  drain_after_timeout(sh.full, timed_out, kstop, nchunks, nst, nst - 2);
  // ---- partials
  float ls = l_run, zl = z_run;
  ls += __shfl_xor_sync(0xffffffffu, ls, 1);
  ls += __shfl_xor_sync(0xffffffffu, ls, 2);
  zl += __shfl_xor_sync(0xffffffffu, zl, 1);
  zl += __shfl_xor_sync(0xffffffffu, zl, 2);
  if (t4 == 0) {
    sh.lsum[warp][g8] = ls;
    sh.zsum[warp][g8] = zl;
  }
  if (warp == 0 && t4 == 0) sh.mfin[g8] = m_run;
  __syncthreads();
  float* ml = reinterpret_cast<float*>(ws + L.ml);
  float* accw = reinterpret_cast<float*>(ws + L.acc);
  if (g8 < G) {
    float zt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) zt += sh.zsum[w][g8];
    // columns 2 t4 and 2 t4 + 1 of n-tile cbk are coordinates warp CPW + (2 t4) CB + cbk and
    // warp CPW + (2 t4 + 1) CB + cbk
    float v0[CB], v1[CB];
#pragma unroll
    for (int cbk = 0; cbk < CB; ++cbk) {
      v0[cbk] = (accv[cbk][0] + accv[cbk][2]) + zt;
      v1[cbk] = (accv[cbk][1] + accv[cbk][3]) + zt;
    }
    float* dst = accw + ((head0 + g8) * st + s) * D + warp * CPW + 2 * t4 * CB;
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
