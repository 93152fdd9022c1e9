// 4-bit key scan with deterministic score bounds, shared by a GQA group.
//
// picx.dev summary, "Algorithm Components" 4: the keys' 4-bit codes (per
// block and channel) bound every score from above, deterministically
// (u_i >= s_i); readsearch.ai "Abstract": one scan over every key serves
// the whole GQA group.  One CTA scans a tile of 256 keys (four 64-token
// blocks) of one (sequence, KV head) for all G query heads:
//   1. the packed codes (256 x d/2 bytes) and the four blocks' (m_c, Delta_c)
//      are staged in shared memory: the codes (d = 128) by one bulk tensor
//      copy completing on an mbarrier, the bounds with cp.async;
//   2. per (block, head) the query is coded to int8 with a residual and a
//      key-rounding slack (16 threads per (block, head), adjacent-pair float32
//      trees over the channels);
//   3. per key, the exact integer dot product I of the 4-bit codes with the
//      int8 query code comes from u8 x s8 tensor-core products (mma.sync
//      m16n8k32: 16 keys x heads x 32 channels, low and high nibbles as
//      bytes), and ubar = fl(fl(alpha I) + b_hi), l = fl(fl(alpha I) + b_lo);
//   4. ubar is stored key-major with the G heads interleaved, and the per-head
//      maxima of l (c*_lo) and ubar are folded into global atomics (the
//      tile's own maximum of ubar is stored per head as well).
#include "csa_args.cuh"

namespace csa {

// Adjacent-pair tree over the CPT values a thread holds, then over 16 lanes.
template <int CPT>
__device__ __forceinline__ float tree16(const float* v) {
  float s;
  if (CPT == 8) {
    s = fadd(fadd(fadd(v[0], v[1]), fadd(v[2], v[3])), fadd(fadd(v[4], v[5]), fadd(v[6], v[7])));
  } else {
    s = fadd(fadd(v[0], v[1]), fadd(v[2], v[3]));
  }
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) s = fadd(s, __shfl_xor_sync(0xffffffffu, s, o));
  return s;
}

// TWO: query codes of two s8 digits, at = 256 hi + lo with |at| <= 127 * 257,
// and the closed-form residual term fl(fl(15 d) * fl(alpha * (1/2 + 2^-6)))
// in place of the two residual trees (|a_c - alpha at_c| <= alpha (1/2 +
// 2^-6) for codes this fine); I = 256 I_hi + I_lo from two products.
// TMA: the code tile arrives by one bulk tensor copy (64-byte swizzle,
// completing on an mbarrier) instead of 16-byte cp.async (plain d = 128
// scan only).
template <int D, int G, typename E, bool TWO, bool REQ, bool DP4A = false, bool TMA = false>
__global__ void __launch_bounds__(256, REQ ? 6 : 0) scan_kernel(const ScanArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                                const __grid_constant__ CUtensorMap tm_codes) {
  static_assert(!TMA || (D == 128 && !TWO && !REQ && !DP4A), "bulk tensor staging: plain d = 128 scan");
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  constexpr int ND = TWO ? 2 : 1;    // query-code digits
  constexpr float QMF = TWO ? 32639.0f : 127.0f;
  constexpr int CPT = D / 16;        // channels per prep thread
  constexpr int ROWB = D / 2;        // bytes of codes per key
  constexpr int CHR = ROWB / 16;     // 16-byte chunks per key
  constexpr int WE = D / 8;          // even (and odd) code words per key
  __shared__ __align__(1024) uint8_t s_codes[kTile * ROWB];
  __shared__ __align__(8) unsigned long long s_bar;   // the code tile's copy (TMA)
  __shared__ __align__(16) float s_bnd[4][2][D];
  __shared__ __align__(16) float s_qt[G][D];
  __shared__ __align__(16) unsigned s_atw[ND][4][G][2 * WE];   // [digit]: lo, hi
  __shared__ float s_q1[G];
  __shared__ float s_alpha[4][G], s_bhi[4][G], s_blo[4][G];
  __shared__ float s_red[8][G][2];

  const int tid = threadIdx.x;
  const int bg = blockIdx.y;
  const int b = bg / a.Hkv;
  const int g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  const int64_t key0 = (int64_t)blockIdx.x * kTile;
  if (key0 >= n) return;
  const int64_t nblk_n = (n + kBlock - 1) / kBlock;
  if (REQ) {
    // the appended token's block, rebuilt before this tile is staged
    __shared__ float s_qvm[kBlock];
    const int64_t lb = (n - 1) / kBlock;
    if (lb * kBlock >= key0 && lb * kBlock < key0 + kTile) {
      const ReqPtrs& rp = *reinterpret_cast<const ReqPtrs*>(a.seqd + 1);
      quantize_block<D, E>(rp.K, rp.V, rp.K4, rp.bounds, rp.vmax, rp.vnorm2, a.n_max, a.nblk_max, bg, lb, n, s_qvm);
      __threadfence();   // the new codes and bounds reach L2 before the copies below read them
      __syncthreads();
    }
  }

  // 1. stage the block bounds (first group: the query prep needs them) and
  // the codes (second group, or the bulk tensor copy: the dot products need
  // them)
  // (the copy's swizzle pattern follows shared-memory address bits: the tile
  // must start on a 1024-byte boundary, else the cp.async staging is taken)
  const bool tma = TMA && (smem_u32(s_codes) & 1023u) == 0u;
  if (tma && tid == 0) {
    mbar_init(smem_u32(&s_bar), 1);
    fence_barrier_init();
  }
  {
    const int64_t blk0 = key0 / kBlock;
    const float* bsrc = a.bounds + ((int64_t)bg * a.nblk_max + blk0) * 2 * D;
    for (int c = tid; c < 4 * 2 * D / 4; c += 256) {
      int blk = c / (2 * D / 4);
      bool ok = blk0 + blk < nblk_n;
      cp_async16(reinterpret_cast<float*>(s_bnd) + c * 4, ok ? bsrc + (int64_t)c * 4 : a.bounds, ok);
    }
    cp_async_commit();
    if (tma) {
      // rows past the group's last block hold other codes (or zeros past
      // the array); they belong to keys >= n, whose bounds are never kept
      __syncthreads();   // the barrier is initialised before anyone waits on it
      if (tid == 0) {
        mbar_expect_tx(smem_u32(&s_bar), (unsigned)(kTile * ROWB));
        tma_load_2d(smem_u32(s_codes), &tm_codes, 0, (int)((int64_t)bg * a.nblk_max * kBlock + key0),
                    smem_u32(&s_bar));
      }
    } else {
      const uint8_t* src = a.K4 + ((int64_t)bg * a.nblk_max * kBlock + key0) * ROWB;
      const int64_t rows_valid = nblk_n * kBlock - key0;
#pragma unroll
      for (int c = tid; c < kTile * CHR; c += 256) {
        const int row = c / CHR, part = c - row * CHR;
        bool ok = row < rows_valid;
        // chunk `part` of a row at chunk part ^ (row % CHR): the fragment
        // loads of eight rows then spread over the banks
        cp_async16(s_codes + row * ROWB + ((part ^ (row & (CHR - 1))) << 4),
                   ok ? src + (int64_t)c * 16 : a.K4, ok);
      }
      cp_async_commit();
    }
  }
  // query (scaled by 1/sqrt d) for the group's G heads
  {
    const E* qp = reinterpret_cast<const E*>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * G) * D;
    bool bad = false;
    for (int i = tid; i < G * D; i += 256) {
      float v = Elem<E>::get(qp, i);
      bad |= !isfinite(v);
      s_qt[i / D][i % D] = fmul(v, a.rs);
    }
    if (bad) atomicOr(a.status, 1u);
  }
  __syncthreads();
  {
    const int w = tid >> 5, lane = tid & 31;
    if (w < G) {
      constexpr int CPL = D / 32;
      float p[CPL];
#pragma unroll
      for (int k = 0; k < CPL; ++k) p[k] = fabsf(s_qt[w][lane * CPL + k]);
      float s = local_tree<CPL>(p);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) s = fadd(s, __shfl_xor_sync(0xffffffffu, s, o));
      if (lane == 0) s_q1[w] = s;
    }
  }
  if (tma) cp_async_wait<0>();   // the bounds group has landed
  else cp_async_wait<1>();
  __syncthreads();

  // 2. per (block, head) query code
  for (int u = tid >> 4; u < 4 * G; u += 16) {
    const int blk = u / G, h = u - blk * G;
    const int l16 = tid & 15;
    const int c0 = l16 * CPT;
    float av[CPT], mv[CPT];
    float amax = 0.f, kabs = 0.f;
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      float dl = s_bnd[blk][1][c0 + k];
      mv[k] = s_bnd[blk][0][c0 + k];
      av[k] = fmul(s_qt[h][c0 + k], dl);
      amax = fmaxf(amax, fabsf(av[k]));
      kabs = fmaxf(kabs, fadd(fabsf(mv[k]), fmul(16.0f, dl)));
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      kabs = fmaxf(kabs, __shfl_xor_sync(0xffffffffu, kabs, o));
    }
    float alpha = 0.f, inv = 0.f;
    if (amax > 0.f) {
      alpha = fdiv(amax, QMF);
      inv = fdiv(QMF, amax);
    }
    float tb[CPT], ta[CPT], tp[CPT], tn[CPT];
    int at[CPT];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      float x = rintf(fmul(av[k], inv));
      x = fminf(fmaxf(x, -QMF), QMF);
      at[k] = (int)x;
      tb[k] = fmul(s_qt[h][c0 + k], mv[k]);
      ta[k] = fabsf(av[k]);
      if (!TWO) {
        float r = fsub(av[k], fmul(alpha, x));
        tp[k] = fmaxf(r, 0.0f);
        tn[k] = fmaxf(-r, 0.0f);
      }
    }
    float Bq = tree16<CPT>(tb);
    float A1 = tree16<CPT>(ta);
    float Rp = 0.f, Rn = 0.f;
    if (!TWO) {
      Rp = tree16<CPT>(tp);
      Rn = tree16<CPT>(tn);
    }
    if (l16 == 0) {
      float sk = fmul(A1, 0.5000152587890625f);
      float hi, lo;
      if (TWO) {
        const float res = fmul((float)(15 * D), fmul(alpha, 0.515625f));
        hi = fadd(sk, res);
        lo = fadd(sk, res);
      } else {
        hi = fadd(sk, fmul(15.0f, Rp));
        lo = fadd(sk, fmul(15.0f, Rn));
      }
      float mag = fadd(fadd(fmul(s_q1[h], kabs), hi), lo);
      float marg = fmul(mag, 6.103515625e-05f);      // 2^-14
      float bhi = fadd(fadd(Bq, hi), marg);
      float blo = fsub(fsub(Bq, lo), marg);
      s_alpha[blk][h] = alpha;
      s_bhi[blk][h] = bhi;
      s_blo[blk][h] = blo;
      // half width of the block's score interval: the candidate pass takes
      // ubar minus it as a score estimate for the stop prediction
      const int64_t gblk = key0 / kBlock + blk;
      if (gblk < nblk_n) a.hw[((int64_t)bg * a.nblk_max + gblk) * G + h] = fmul(0.5f, fsub(bhi, blo));
      if (!isfinite(bhi) || !isfinite(blo) || !isfinite(alpha)) atomicOr(a.status, 1u);
    }
    // pack the code (each digit): word w covers channels 8w..8w+7; even
    // word = channels 8w, 8w+2, 8w+4, 8w+6 (bytes 0..3), odd word = 8w+1,
    // ..., 8w+7.  Two digits: hi = floor((at + 128) / 256) in [-127, 127],
    // lo = at - 256 hi in [-128, 127].
#pragma unroll
    for (int dd = 0; dd < ND; ++dd) {
      int dg[CPT];
#pragma unroll
      for (int k = 0; k < CPT; ++k) {
        const int hi = (at[k] + 128) >> 8;      // arithmetic shift: floor
        dg[k] = !TWO ? at[k] : (dd == 0 ? at[k] - 256 * hi : hi);
      }
      if (CPT == 8) {
        unsigned ev = (dg[0] & 0xFF) | ((dg[2] & 0xFF) << 8) | ((dg[4] & 0xFF) << 16) | ((unsigned)(dg[6] & 0xFF) << 24);
        unsigned od = (dg[1] & 0xFF) | ((dg[3] & 0xFF) << 8) | ((dg[5] & 0xFF) << 16) | ((unsigned)(dg[7] & 0xFF) << 24);
        s_atw[dd][blk][h][l16] = ev;
        s_atw[dd][blk][h][WE + l16] = od;
      } else {
        unsigned short ev = (unsigned short)((dg[0] & 0xFF) | ((dg[2] & 0xFF) << 8));
        unsigned short od = (unsigned short)((dg[1] & 0xFF) | ((dg[3] & 0xFF) << 8));
        reinterpret_cast<unsigned short*>(&s_atw[dd][blk][h][0])[l16] = ev;
        reinterpret_cast<unsigned short*>(&s_atw[dd][blk][h][WE])[l16] = od;
      }
    }
  }
  if (tma) {
    // the codes too (bounded wait; on a timeout the CTA records it, waits
    // once more for its copy and leaves)
    const bool ok = mbar_wait(smem_u32(&s_bar), 0);
    if (!__syncthreads_and(ok)) {
      if (tid == 0) atomicOr(a.status, 4u);
      mbar_wait(smem_u32(&s_bar), 0);
      return;
    }
  } else {
    cp_async_wait<0>();          // the codes too
    __syncthreads();
  }

  // 3. bounds per key.  The exact integer dot products I = sum_c qcode_c *
  // code_c come from u8 x s8 m16n8k32 tensor-core products: a warp takes its
  // 32 keys (one 64-key block) as two 16-key tiles (M), the heads are N
  // (padded to 8), and k-step s covers code words 4s..4s+3: thread t's four
  // k positions 4t..4t+3 are the even channels of word 4s+t (low nibbles)
  // and 16+4t..16+4t+3 its odd channels (high nibbles), matching the even
  // and odd query-code words.  Integer sums are exact in any order.
  const int w = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int blk = w >> 1;
  constexpr int KS = D / 32;
  unsigned bq[ND][KS][2];
#pragma unroll
  for (int dd = 0; dd < ND; ++dd)
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      bq[dd][ks][0] = gq < G ? s_atw[dd][blk][gq < G ? gq : 0][4 * ks + tq] : 0u;
      bq[dd][ks][1] = gq < G ? s_atw[dd][blk][gq < G ? gq : 0][WE + 4 * ks + tq] : 0u;
    }
  float lmax[2] = {-INFINITY, -INFINITY}, umax[2] = {-INFINITY, -INFINITY};   // heads 2tq, 2tq+1
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = 32 * w + 16 * mt + gq, r1 = r0 + 8;
    int acc[ND][4];
#pragma unroll
    for (int dd = 0; dd < ND; ++dd) acc[dd][0] = acc[dd][1] = acc[dd][2] = acc[dd][3] = 0;
#pragma unroll
    for (int ks = 0; ks < (DP4A ? 0 : KS); ++ks) {
      // word 4ks+tq of rows r0, r1: chunk ks, word tq (swizzled chunks)
      // (the bulk tensor copy's 64-byte swizzle puts chunk c of row r at
      // c ^ ((r / 2) % 4); the cp.async staging at c ^ (r % CHR))
      const int s0 = tma ? ((r0 >> 1) & 3) : (r0 & (CHR - 1));
      const int s1 = tma ? ((r1 >> 1) & 3) : (r1 & (CHR - 1));
      const unsigned w0 = *reinterpret_cast<const unsigned*>(s_codes + r0 * ROWB + ((ks ^ s0) << 4) + 4 * tq);
      const unsigned w1 = *reinterpret_cast<const unsigned*>(s_codes + r1 * ROWB + ((ks ^ s1) << 4) + 4 * tq);
      const unsigned af0 = w0 & 0x0F0F0F0Fu, af1 = w1 & 0x0F0F0F0Fu;
      const unsigned af2 = (w0 >> 4) & 0x0F0F0F0Fu, af3 = (w1 >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int dd = 0; dd < ND; ++dd)
        asm volatile(
            "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+r"(acc[dd][0]), "+r"(acc[dd][1]), "+r"(acc[dd][2]), "+r"(acc[dd][3])
            : "r"(af0), "r"(af1), "r"(af2), "r"(af3), "r"(bq[dd][ks][0]), "r"(bq[dd][ks][1]));
    }
    // I = 256 I_hi + I_lo (|I| < 2^26: exact in int32)
    int I4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) I4[e] = TWO ? acc[ND - 1][e] * 256 + acc[0][e] : acc[0][e];
    if constexpr (DP4A) {
      // the CUDA-core alternative for the same (key, head) pairs: dp4a over
      // the code words, low nibbles (even channels) with the even query
      // word, high nibbles with the odd one (kept to compare the two)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e < 2 ? r0 : r1, h = 2 * tq + (e & 1);
        int sacc = 0;
        if (h < G) {
#pragma unroll
          for (int k = 0; k < WE; ++k) {
            const unsigned wv = *reinterpret_cast<const unsigned*>(
                s_codes + r * ROWB + (((k >> 2) ^ (r & (CHR - 1))) << 4) + 4 * (k & 3));
            sacc = __dp4a((int)(wv & 0x0F0F0F0Fu), (int)s_atw[0][blk][h][k], sacc);
            sacc = __dp4a((int)((wv >> 4) & 0x0F0F0F0Fu), (int)s_atw[0][blk][h][WE + k], sacc);
          }
        }
        I4[e] = sacc;
      }
    }
    // acc[0], acc[1]: key r0, heads 2tq, 2tq+1; acc[2], acc[3]: key r1
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? r1 : r0;
      const int64_t key = key0 + r;
      const bool live = key < n;
      float ubv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int h = 2 * tq + u;
        ubv[u] = 0.f;
        if (h < G) {
          const float aI = fmul(s_alpha[blk][h], (float)I4[2 * half + u]);
          const float ub = fadd(aI, s_bhi[blk][h]);
          const float lo = fadd(aI, s_blo[blk][h]);
          ubv[u] = ub;
          if (live) { umax[u] = fmaxf(umax[u], ub); lmax[u] = fmaxf(lmax[u], lo); }
        }
      }
      if (live && 2 * tq < G) {
        float* dst = a.ubar + ((int64_t)bg * a.n_max + key) * G + 2 * tq;
        if (G >= 2) *reinterpret_cast<float2*>(dst) = make_float2(ubv[0], ubv[1]);
        else dst[0] = ubv[0];
      }
    }
  }
  // 4. per-head maxima: over the eight key rows of the thread's column
  // group, then over the warps
#pragma unroll
  for (int u = 0; u < 2; ++u) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lmax[u] = fmaxf(lmax[u], __shfl_xor_sync(0xffffffffu, lmax[u], o));
      umax[u] = fmaxf(umax[u], __shfl_xor_sync(0xffffffffu, umax[u], o));
    }
  }
  if (gq == 0) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int h = 2 * tq + u;
      if (h < G) { s_red[w][h][0] = lmax[u]; s_red[w][h][1] = umax[u]; }
    }
  }
  __syncthreads();
  if (tid < G) {
    float x = -INFINITY, y = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) { x = fmaxf(x, s_red[i][tid][0]); y = fmaxf(y, s_red[i][tid][1]); }
    unsigned* slot = a.cmax + ((int64_t)b * a.Hq + (int64_t)g * G + tid) * 4;
    if (x > -INFINITY) atomic_max_f(slot + 0, x);
    if (y > -INFINITY) atomic_max_f(slot + 1, y);
    // the tile's largest ubar: the exact-max pass skips tiles below c*_lo
    a.tmax[((int64_t)bg * ((a.n_max + kTile - 1) / kTile) + blockIdx.x) * G + tid] = y;
  }
}

template <int D, int G, typename E>
cudaError_t launch_scan_t(const ScanArgs& a, const SeqArgs& seq, int B, int64_t nmax_live, const CUtensorMap* tm,
                          cudaStream_t st) {
  dim3 grid((unsigned)((nmax_live + kTile - 1) / kTile), (unsigned)(B * a.Hkv));
  static const CUtensorMap none = {};
  const CUtensorMap& t = tm ? *tm : none;
  // REQ: the variant that re-quantises the appended block first (device-
  // length steps); a separate instantiation keeps the plain scan's
  // registers (and resident CTAs) as they are
  if (a.dp4a && !a.requant && !a.two_digit) {
    launch_pdl(scan_kernel<D, G, E, false, false, true>, grid, dim3(256), 0, st, a, seq, t);
  } else if (a.requant) {
    if (a.two_digit) launch_pdl(scan_kernel<D, G, E, true, true>, grid, dim3(256), 0, st, a, seq, t);
    else launch_pdl(scan_kernel<D, G, E, false, true>, grid, dim3(256), 0, st, a, seq, t);
  } else if (a.two_digit) {
    launch_pdl(scan_kernel<D, G, E, true, false>, grid, dim3(256), 0, st, a, seq, t);
  } else if constexpr (D == 128) {
    if (tm) launch_pdl(scan_kernel<D, G, E, false, false, false, true>, grid, dim3(256), 0, st, a, seq, t);
    else launch_pdl(scan_kernel<D, G, E, false, false>, grid, dim3(256), 0, st, a, seq, t);
  } else {
    launch_pdl(scan_kernel<D, G, E, false, false>, grid, dim3(256), 0, st, a, seq, t);
  }
  return cudaGetLastError();
}

#define CSA_SCAN_CASE(DD, GG)                                                          \
  if (d == DD && G == GG)                                                              \
    return bf16 ? launch_scan_t<DD, GG, __nv_bfloat16>(a, seq, B, nmax_live, tm, st)   \
                : launch_scan_t<DD, GG, float>(a, seq, B, nmax_live, tm, st);

cudaError_t launch_scan(const ScanArgs& a, const SeqArgs& seq, int B, int d, int G, bool bf16,
                        int64_t nmax_live, const CUtensorMap* tm, cudaStream_t st) {
  CSA_SCAN_CASE(128, 1) CSA_SCAN_CASE(128, 2) CSA_SCAN_CASE(128, 4) CSA_SCAN_CASE(128, 8)
  CSA_SCAN_CASE(64, 1) CSA_SCAN_CASE(64, 2) CSA_SCAN_CASE(64, 4) CSA_SCAN_CASE(64, 8)
  return cudaErrorInvalidValue;
}

}  // namespace csa
