// The sparse part of the decode step, after the 4-bit scan.
//
// picx.dev summary, "Algorithm Components" 1-4 and Theorem 4; readsearch.ai
// "Abstract".  Kernels, in launch order, for every (sequence b, KV head g):
//   cset_kernel     the exact-max set: the window and the pool keys with
//                   ubar >= c*_lo for some head, compacted into a list
//   rows_kernel<0>  float32 rescoring of the listed K rows (one row load
//                   serves the G heads): c32 = max score and the certified
//                   lower bound cb = max fl(s32 - fl(mag * 2^-13))
//   cand_kernel     perturbations t_i, bound levels jbar_i, candidates
//                   (jbar <= J); keys of the exact-max set keep the scores
//                   already computed, the others are compacted into a list;
//                   per-level counts and heavy weights of estimated levels
//                   (no values, no K rows: for the stop predictor)
//   predict_kernel  window sums (D_R, N_R, H_R) and a predicted stop level
//                   per head that sizes the first gather round
//   rows_kernel<1>  (per round) float32 scores of the listed candidates
//                   whose smallest bound level lies in the range that the
//                   round's levels newly need (jbar_i <= j implies
//                   jl_i >= jbar_i, so a key outside it has no event there)
//   levels_kernel   (per round) each key that changes a head's sums at a
//                   level of the round is appended once to the (b, g, level)
//                   bucket, with per-head event masks
//   vplan_kernel    (per round, only for large batches) ranges of the new
//                   bucket entries (otherwise each value-sum CTA computes
//                   them)
//   vsum_kernel     (per round, bf16) V rows of the bucketed keys in
//                   batches of 16 entries of one level; per-level
//                   Horvitz-Thompson sums (light count, sum v, sum ||v||^2;
//                   heavy sum w, sum w v, sum w ||v||^2) per head as
//                   tensor-core products (vgather_kernel: the float32 path)
//   certify_kernel  (per round) prefix over levels, Chernoff interval,
//                   Bernstein bound on G, Pinelis bound zeta, beta, value
//                   scale lower bound; first certified level -> outputs;
//                   a head with none in its range goes to the next round
//   near_kernel     optional diagnostics: near-threshold keys at the stop,
//                   rows read per group
// Row gathers (K rows, V rows) go through a per-warp ring of shared-memory
// stages filled with cp.async, so the bytes in flight do not depend on the
// registers a thread holds.
#include "csa_args.cuh"

namespace csa {

constexpr int kFlagFallback = 1;
constexpr int kFlagDone = 2;
constexpr int kChunk = 1024;   // bucket entries per gather work item
// Work units a non-empty bucket costs beyond its entries (its partial batch
// and the flush of its sums): the warps' shares are equal in entries plus
// this per bucket, so a warp whose range crosses many small buckets (the
// deep levels of peaked heads) does not become the launch's straggler.
// (128 x 4 step, value sums of the unsplit chain: 153 us with no bucket
// cost, 132 us with 32 to 128; the split step 674 -> 662 us at 128.)
#ifndef CSA_VS_BUCKET_COST
#define CSA_VS_BUCKET_COST 128
#endif
constexpr unsigned kVsBucketCost = CSA_VS_BUCKET_COST;
#ifndef CSA_RING_S
#define CSA_RING_S 4
#endif
#ifndef CSA_RING_W
#define CSA_RING_W 4
#endif
#ifndef CSA_ROWS_CPS
#define CSA_ROWS_CPS 16
#endif
#ifndef CSA_ROWS0_CPS
#define CSA_ROWS0_CPS 5
#endif
constexpr int kRingS = CSA_RING_S;   // ring stages per warp (8 rows each)
constexpr int kRingW = CSA_RING_W;   // warps per CTA of the ring kernels
constexpr int kRowsCps = CSA_ROWS_CPS;   // ring CTAs launched per SM (candidate rounds)
constexpr int kRows0Cps = CSA_ROWS0_CPS; // the same for the (small) exact-max set: one wave
                                         // (128K x 4 step: 656 us against 662 us at 12)

// ----------------------------------------------------------- small helpers

template <int D, typename E>
__device__ __forceinline__ void load_row(const E* row, float* v) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  if (CPL == 4) {
    float4 f = Elem<E>::get4(row + lane * 4);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else {
    float2 f = Elem<E>::get2(row + lane * 2);
    v[0] = f.x; v[1] = f.y;
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float cmax_get(const SparseArgs& a, int bh, int k) {
  return float_of_ord(a.cmax[(int64_t)bh * 4 + k]);
}

// Round queues: the (sequence, KV head) groups that take part in gather
// round r, each listed once (rq layout in SparseArgs).
__device__ __forceinline__ void rq_push(const SparseArgs& a, int r, int bg) {
  const int BG = a.B * a.Hkv;
  if (atomicOr(a.rq + 3 * BG + r * BG + bg, 1u) == 0u) {
    const unsigned i = atomicAdd(a.rq + 6 * BG + r, 1u);
    a.rq[r * BG + i] = (unsigned)bg;
  }
}

// Warp-aggregated append of this lane's item to a global list (lanes with
// want = false take no slot).  Returns the slot or -1.
__device__ __forceinline__ int warp_append(unsigned* counter, bool want) {
  const int lane = threadIdx.x & 31;
  const unsigned bal = __ballot_sync(0xffffffffu, want);
  unsigned base = 0;
  if (lane == 0 && bal) base = atomicAdd(counter, (unsigned)__popc(bal));
  base = __shfl_sync(0xffffffffu, base, 0);
  return want ? (int)(base + __popc(bal & ((1u << lane) - 1u))) : -1;
}


// phi(y) = e^y - 1 - y from y and expm1(y) (a series near 0, where
// expm1(y) - y cancels)
__device__ __forceinline__ float phi_em1(float y, float em1) {
  if (fabsf(y) < 0.05f) return y * y * (0.5f + y * (1.0f / 6.0f + y * (1.0f / 24.0f + y * (1.0f / 120.0f))));
  return em1 - y;
}

// Chernoff interval for a Poisson-binomial count k (two-sided, budget
// delta_e / 2 per side): mu = k e^y with phi(y) = Lz / k.  Returns
// k - mu_lo and mu_hi - k (both >= 0).  phi is convex, so Newton's
// iteration started outside a root (where phi > Lz / k) stays outside and
// converges to it monotonically: the iterates are outward ends of the
// root's bracket, as the certificate needs.  Each step takes one expm1:
// its value at the new iterate is both that iterate's phi and the next
// step's slope.
__device__ void chernoff_gaps(float k, float Lz, float& below, float& above) {
  if (!(k > 0.f)) { below = 0.f; above = Lz; return; }
  const float c0 = Lz / k;
  // upper root: start where phi >= c0, step down the tangent.  phi(y) >=
  // y^2 / 2 for y >= 0, so sqrt(2 c0) lies at or past the root (within a
  // few per cent of it for small c0: large counts then converge in one to
  // three steps instead of about ten)
  const float s2 = sqrtf(2.0f * c0);
  float hi = fminf(s2, fmaxf(1.0f, logf(3.0f * c0 + 3.0f)));
  float eh = expm1f(hi), ph = phi_em1(hi, eh);
  for (int it = 0; it < 8 && ph < c0; ++it) {
    hi *= 2.0f;
    eh = expm1f(hi);
    ph = phi_em1(hi, eh);
  }
  for (int it = 0; it < 12; ++it) {
    const float nx = hi - (ph - c0) / eh;
    if (!(nx < hi)) break;                        // converged
    const float en = expm1f(nx), pn = phi_em1(nx, en);
    if (pn < c0) break;                           // rounding crossed the root
    hi = nx; eh = en; ph = pn;
  }
  above = k * eh;
  // lower root: start at -(sqrt(2 c0) + c0) when phi >= c0 there (the
  // root lies near -(sqrt(2 c0) + c0 / 3) for small c0), else at -(c0 + 1)
  // (phi > c0 always); step up the tangent
  float lo = -(s2 + c0);
  float el = expm1f(lo), pl = phi_em1(lo, el);
  if (!(pl >= c0)) {
    lo = -(c0 + 1.0f);
    el = expm1f(lo);
    pl = phi_em1(lo, el);
  }
  for (int it = 0; it < 12; ++it) {
    const float nx = lo - (pl - c0) / el;
    if (!(nx > lo) || nx >= 0.f) break;
    const float en = expm1f(nx), pn = phi_em1(nx, en);
    if (pn < c0) break;
    lo = nx; el = en; pl = pn;
  }
  below = -k * el;
}

// Stage eight rows (row indices ent[0..nvalid).x) of a [rows][D] array into
// dst with 16-byte cp.async copies; missing rows are zero-filled.
template <int D, typename E>
__device__ __forceinline__ void stage8(uint8_t* dst, const E* base, const uint2* ent, int nvalid) {
  constexpr int RB = D * (int)sizeof(E);
  constexpr int CH = RB / 16;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = lane; c < 8 * CH; c += 32) {
    const int r = c / CH, part = c - r * CH;
    const bool ok = r < nvalid;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(base) + (ok ? (int64_t)ent[r].x * RB + part * 16 : 0);
    cp_async16(dst + r * RB + part * 16, src, ok);
  }
}

// NB rows with the 16-byte chunk c of row r stored at chunk c ^ (r & 7)
// (tensor-core fragment loads of eight rows then hit eight bank groups).
template <int D, typename E, int NB>
__device__ __forceinline__ void stage_swz(uint8_t* dst, const E* base, const uint2* ent, int nvalid) {
  constexpr int RB = D * (int)sizeof(E);
  constexpr int CH = RB / 16;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = lane; c < NB * CH; c += 32) {
    const int r = c / CH, part = c - r * CH;
    const bool ok = r < nvalid;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(base) + (ok ? (int64_t)ent[r].x * RB + part * 16 : 0);
    cp_async16(dst + r * RB + ((part ^ (r & 7)) * 16), src, ok);
  }
}

__device__ __forceinline__ void ldsm_x4(unsigned (&r)[4], const void* p) {
  unsigned sa = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(sa));
}


__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const unsigned (&a)[4], unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------------------- exact-max set

#ifndef CSA_CSET_TILES
#define CSA_CSET_TILES 16
#endif
constexpr int kCsetTiles = CSA_CSET_TILES;   // 256-key tiles per exact-max-set CTA (at most 16: static list)
static_assert(kCsetTiles % 4 == 0 && kCsetTiles <= 16, "tiles are read four at a time; the list is static");

// A CTA covers `span` keys (kCsetTiles 256-key tiles) of one group.  A
// pool tile whose largest ubar (per head, from the scan) lies below c*_lo
// for every head holds no member and is not read; the others are read four
// tiles at a time.
template <int G>
__global__ void __launch_bounds__(256) cset_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                   int span) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  // members are staged in shared memory and take one slot range of the
  // group's list per CTA (a per-warp reservation on the group's counter
  // serialises)
  __shared__ uint2 s_list[256 * kCsetTiles];
  __shared__ unsigned s_n, s_live;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  const int64_t k0 = (int64_t)blockIdx.x * span;
  if (k0 >= n) return;
  const int64_t kstop = min(n, k0 + span);
  const int bh0 = b * a.Hq + g * G;
  float clo[G];
#pragma unroll
  for (int h = 0; h < G; ++h) clo[h] = cmax_get(a, bh0 + h, 0);
  // tiles that may hold a member: warp 0, lane = tile
  if (threadIdx.x < 32) {
    const int64_t kt = k0 + (int64_t)threadIdx.x * kTile;
    bool live = false;
    if (threadIdx.x < kCsetTiles && kt < kstop) {
      if (kt + kTile > P) live = true;                 // window keys are members
      else {
        const float* tm = a.tmax + ((int64_t)bg * ((a.n_max + kTile - 1) / kTile) + kt / kTile) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) live |= tm[h] >= clo[h];
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, live);
    if (threadIdx.x == 0) { s_live = m; s_n = 0u; }
  }
  __syncthreads();
  const unsigned lm = s_live;
  auto load = [&](int64_t key, float (&u)[G]) {
#pragma unroll
    for (int h = 0; h < G; ++h) u[h] = -INFINITY;
    if (key >= P) return;
    const float* ub = a.ubar + ((int64_t)bg * a.n_max + key) * G;
    if (G == 4) {
      const float4 f = *reinterpret_cast<const float4*>(ub);
      u[0] = f.x; u[1 % G] = f.y; u[2 % G] = f.z; u[3 % G] = f.w;
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) u[h] = ub[h];
    }
  };
  for (int t0 = 0; t0 < kCsetTiles; t0 += 4) {
    if (!((lm >> t0) & 0xFu)) continue;
    float u[4][G];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t key = k0 + (int64_t)(t0 + j) * kTile + threadIdx.x;
      if ((lm >> (t0 + j)) & 1u) load(key, u[j]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!((lm >> (t0 + j)) & 1u)) continue;
      const int64_t key = k0 + (int64_t)(t0 + j) * kTile + threadIdx.x;
      unsigned qm = 0;
      if (key < kstop) {
        if (key >= P) qm = (1u << G) - 1u;
        else {
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (u[j][h] >= clo[h]) qm |= 1u << h;
        }
      }
      const int slot = warp_append(&s_n, qm != 0);
      if (slot >= 0) s_list[slot] = make_uint2((unsigned)key, qm);
    }
  }
  __syncthreads();
  __shared__ unsigned s_gbase;
  if (threadIdx.x == 0) s_gbase = s_n ? atomicAdd(a.xcnt + bg, s_n) : 0u;
  __syncthreads();
  for (unsigned i = threadIdx.x; i < s_n; i += 256) a.xlist[(int64_t)bg * a.n_max + s_gbase + i] = s_list[i];
}

// ------------------------------------------------------ ring row scoring
//
// MODE 0 (exact max): entries = exact-max set.  Scores and |product| sums
//   of every head; the maxima of s32 and fl(s32 - fl(mag 2^-13)) over the
//   heads in the entry's mask; raw scores stored (pool: s32, window: win).
// MODE 1 (candidates, per round): entries = candidates whose smallest bound
//   level lies in (lold, lnew], the range this round newly needs (lnew = the
//   largest range end of the group's heads still running); scores stored,
//   -inf for the heads the key is not a candidate of.
//
// Each warp takes a contiguous share of the list (in key order within the
// candidate pass's CTA chunks, so consecutive rows are mostly adjacent in
// HBM), reads it 128 entries ahead, compacts the wanted entries into a
// small queue and stages them eight rows per ring slot.

constexpr int kQueue = 64;       // per-warp queue of wanted entries (power of 2)

template <int D, int G, typename E>
__host__ __device__ constexpr int rows_smem() {
  return kRingW * kRingS * 8 * D * (int)sizeof(E) + kRingW * kRingS * 8 * 8 + kRingW * kQueue * 8 +
         kRingW * G * 2 * 4;
}

template <int D, int G, typename E, int MODE>
__global__ void __launch_bounds__(kRingW * 32) rows_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                   int round) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  constexpr int CPL = D / 32;
  constexpr int RB = D * (int)sizeof(E);
  extern __shared__ __align__(16) uint8_t dsm[];
  uint8_t* ring = dsm;
  uint2* s_ent = reinterpret_cast<uint2*>(dsm + kRingW * kRingS * 8 * RB);
  uint2* s_q = s_ent + kRingW * kRingS * 8;
  float* s_red = reinterpret_cast<float*>(s_q + kRingW * kQueue);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  const int bh0 = b * a.Hq + g * G;
  const uint2* list;
  int cnt, lold = -1, lnew = -1;
  if (MODE == 0) {
    list = a.xlist + (int64_t)bg * a.n_max;
    cnt = (int)a.xcnt[bg];
  } else {
    list = a.clist + (int64_t)bg * a.pcap;
    cnt = (int)a.ccnt[bg];
    const int BG = a.B * a.Hkv;
    lold = a.front[round * BG + bg] - 1;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int* st = a.state + (int64_t)(bh0 + h) * 4;
      if (!(st[3] & kFlagDone)) lnew = max(lnew, st[1]);
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) a.front[(round + 1) * BG + bg] = max(lold, lnew) + 1;
    if (lnew <= lold) return;
  }
  // the warp's share [cur, end) of the list
  const int nw = gridDim.x * kRingW;
  const int wid = blockIdx.x * kRingW + w;
  int cur = (int)((int64_t)cnt * wid / nw);
  const int end = (int)((int64_t)cnt * (wid + 1) / nw);
  float qv[G][CPL];
  if (MODE == 0 || sizeof(E) != 2) {
    const E* qp = reinterpret_cast<const E*>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * G) * D;
#pragma unroll
    for (int h = 0; h < G; ++h) load_row<D, E>(qp + (int64_t)h * D, qv[h]);
  }
  float cbm[G], c3m[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { cbm[h] = -INFINITY; c3m[h] = -INFINITY; }
  const E* Kb = reinterpret_cast<const E*>(a.K) + (int64_t)bg * a.n_max * D;
  constexpr bool TC = (MODE == 1) && (sizeof(E) == 2);   // tensor-core scoring
  // rows per ring slot and slots per warp (the same shared memory either
  // way): the tensor-core path scores 16 rows per product chain
  constexpr int NB = TC ? 16 : 8;
  constexpr int NS = TC ? kRingS / 2 : (kRingS < 4 ? kRingS : 4);
  static_assert(NB * NS <= 8 * kRingS && NS >= 2 && NS <= 4, "ring size (slot counts are packed 8 bits each)");
  uint8_t* my = ring + w * kRingS * 8 * RB;
  uint2* me = s_ent + w * kRingS * 8;
  uint2* myq = s_q + w * kQueue;
  // entries are read 128 at a time (four per lane), one window ahead
  uint2 cw[4], nx[4];
  auto load_win = [&](int base, uint2 (&dst)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = base + 32 * k + lane;
      dst[k] = i < end ? list[i] : make_uint2(~0u, 0u);
    }
  };
  load_win(cur, cw);
  load_win(cur + 128, nx);
  int ck = 0;                 // next 32-entry chunk of the current window
  int qh = 0, qt = 0;         // queue head and tail (warp-uniform)
  // fill ring slot k with up to NB wanted entries; 0 only when the warp's
  // share is exhausted
  auto produce = [&](int k) {
    while (qt - qh < NB && cur < end) {
      const uint2 e = ck == 0 ? cw[0] : (ck == 1 ? cw[1] : (ck == 2 ? cw[2] : cw[3]));
      bool keep = e.x != ~0u;
      if (MODE == 1 && keep) {
        const int jm = a.refine8 ? (int)(a.jkey[(int64_t)bg * a.pcap + e.x] & 0x1FFu) : (int)((e.y >> 8) & 0xFFu);
        keep = jm > lold && jm <= lnew;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      if (keep) myq[(qt + __popc(bal & ((1u << lane) - 1u))) & (kQueue - 1)] = e;
      qt += __popc(bal);
      cur += 32;
      if (++ck == 4) {
        ck = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) cw[q] = nx[q];
        load_win(cur + 128, nx);
      }
    }
    __syncwarp();
    const int take = min(NB, qt - qh);
    if (lane < take) me[k * NB + lane] = myq[(qh + lane) & (kQueue - 1)];
    qh += take;
    __syncwarp();
    return take;
  };
  auto stage = [&](int k, int nv) {
    if (TC) stage_swz<D, E, NB>(my + k * NB * RB, Kb, me + k * NB, nv);
    else stage8<D, E>(my + k * NB * RB, Kb, me + k * NB, nv);
    cp_async_commit();
  };
  unsigned nvpack = 0;        // rows staged per slot, 8 bits each
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int nv = produce(k);
    nvpack |= (unsigned)nv << (8 * k);
    stage(k, nv);
  }
  // query fragments for the tensor-core path: the B operand (K = channels,
  // N = heads padded to 8), two bf16 per register
  constexpr int KS = D / 16;
  unsigned qa[KS][2];
  if (TC) {
    const int gq = lane >> 2, tq = lane & 3;
    const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q) +
                              ((int64_t)b * a.Hq + (int64_t)g * G + (gq < G ? gq : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qa[ks][0] = gq < G ? *reinterpret_cast<const unsigned*>(qp + 16 * ks + 2 * tq) : 0u;
      qa[ks][1] = gq < G ? *reinterpret_cast<const unsigned*>(qp + 16 * ks + 2 * tq + 8) : 0u;
    }
  }
  for (int it = 0;; ++it) {
    const int slot = it % NS;
    const int nv = (int)((nvpack >> (8 * slot)) & 0xFFu);
    // slots are filled in order, so the first empty one ends the share
    if (nv == 0) break;
    cp_async_wait<NS - 1>();
    __syncwarp();
    if (TC) {
      // scores of the stage's 16 rows for all heads in one chain of
      // m16n8k16 products: A = rows x channels (ldmatrix from the swizzled
      // stage), B = the query heads; lane (g, t) gets rows g and g + 8,
      // heads 2t and 2t + 1 (rows past nv hold zeros and are not stored)
      const int gq = lane >> 2, tq = lane & 3;
      const int lr = (lane & 7) + ((lane >> 3) & 1) * 8;     // row this lane addresses
      const uint8_t* st = my + slot * NB * RB + lr * RB;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int c = 2 * ks + (lane >> 4);                    // 16-byte chunk of channels
        unsigned af[4];
        ldsm_x4(af, st + ((c ^ (lr & 7)) * 16));
        mma_bf16_16816(acc, af, qa[ks][0], qa[ks][1]);
      }
      if (2 * tq < G) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int r = gq + 8 * half;
          if (r < nv) {
            const uint2 en = me[slot * NB + r];
            float* dst = a.s32 + ((int64_t)bg * a.pcap + en.x) * G + 2 * tq;
            const float x0 = ((en.y >> (2 * tq)) & 1u) ? fmul(acc[2 * half], a.rs) : -INFINITY;
            if (G >= 2) {
              const float x1 = ((en.y >> (2 * tq + 1)) & 1u) ? fmul(acc[2 * half + 1], a.rs) : -INFINITY;
              *reinterpret_cast<float2*>(dst) = make_float2(x0, x1);
            } else {
              dst[0] = x0;
            }
          }
        }
      }
    } else {
      float kv[8][CPL];
#pragma unroll
      for (int r = 0; r < 8; ++r) load_row<D, E>(reinterpret_cast<const E*>(my + (slot * 8 + r) * RB), kv[r]);
      float sc[G], mg[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float part[8], pm[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          float p[CPL], pa[CPL];
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            p[c] = fmul(kv[r][c], qv[h][c]);
            pa[c] = fabsf(p[c]);
          }
          part[r] = local_tree<CPL>(p);
          if (MODE == 0) pm[r] = local_tree<CPL>(pa);
        }
        sc[h] = fmul(reduce8_rows(part), a.rs);
        if (MODE == 0) mg[h] = fmul(reduce8_rows(pm), a.rs);
      }
      const int r = lane & 7;
      if (lane < 8 && r < nv) {
        const uint2 en = me[slot * 8 + r];
        const int64_t key = en.x;
        const unsigned cm = en.y;
        if (MODE == 0) {
          float* wp = key >= P ? a.win + ((int64_t)bg * kWindow + (key - P)) * G
                               : a.s32 + ((int64_t)bg * a.pcap + key) * G;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            wp[h] = sc[h];
            if ((cm >> h) & 1u) {
              cbm[h] = fmaxf(cbm[h], fsub(sc[h], fmul(mg[h], 1.220703125e-04f)));   // 2^-13
              c3m[h] = fmaxf(c3m[h], sc[h]);
            }
          }
        } else {
          float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
#pragma unroll
          for (int h = 0; h < G; ++h) sp[h] = ((cm >> h) & 1u) ? sc[h] : -INFINITY;
        }
      }
    }
    __syncwarp();
    // refill this slot: the next rows of the share, kRingS batches ahead
    const int nn = produce(slot);
    nvpack = (nvpack & ~(0xFFu << (8 * slot))) | ((unsigned)nn << (8 * slot));
    stage(slot, nn);
  }
  cp_async_wait<0>();
  if (MODE == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float x = warp_max(cbm[h]), y = warp_max(c3m[h]);
      if (lane == 0) { s_red[(w * G + h) * 2] = x; s_red[(w * G + h) * 2 + 1] = y; }
    }
    __syncthreads();
    if (tid < G) {
      float x = -INFINITY, y = -INFINITY;
      for (int i = 0; i < kRingW; ++i) {
        x = fmaxf(x, s_red[(i * G + tid) * 2]);
        y = fmaxf(y, s_red[(i * G + tid) * 2 + 1]);
      }
      if (x > -INFINITY) atomic_max_f(a.cmax + (int64_t)(bh0 + tid) * 4 + 2, x);
      if (y > -INFINITY) atomic_max_f(a.cmax + (int64_t)(bh0 + tid) * 4 + 3, y);
    }
  }
}

// ------------------------------------------------- 8-bit refinement tier
//
// picx.dev "Algorithm Components" 4: an 8-bit stage between the 4-bit
// candidates and the exact 16-bit reads.  Before a round's rescoring, every
// pool key whose smallest bound level lies in the range the round newly
// needs also gets the upper bound ubar8 from its 8-bit codes (same blocks
// and minima, 255 levels, 12-bit query codes: the 4-bit construction with
// 15 -> 255, 16 -> 256 and QM = 2047), and per head the refined bound level
//   jref = max(0, ceil(fl(fl(-r xbar) - 2^-10))),
//   xbar = fl(fl(fl(min(ubar4, ubar8) - cb) * log2e) + t).
// jbar <= jref <= the exact level, so the sample, the estimates and every
// result stay the same; the key's smallest level over its heads becomes the
// smallest jref, and a key whose jref lies past the round's range waits for
// a later round (or is never read).  keys_read counts jref instead of jbar.
// One warp per 64-key block with a key to refine: it stages the block's
// 8-bit rows of those keys, codes the query per head (one lane per four
// channels, the same adjacent-pair float32 trees as the 4-bit query codes),
// and takes the exact integer dots on tensor cores (u8 codes x two s8
// digits of the 12-bit query codes, mma.sync m16n8k32).
constexpr int kRfW = 4;          // warps per refinement CTA

template <int D, int G>
struct RfLayout {
  static constexpr int rows = 0;                         // [64][D] u8, 16-byte chunks swizzled
  static constexpr int dig = rows + 64 * D;              // [2][8][D] s8 query digits (lo, hi)
  static constexpr int ub8 = dig + 2 * 8 * D;            // [64][8] float ubar8
  static constexpr int per_warp = ub8 + 64 * 8 * 4;
  static constexpr int hist = kRfW * per_warp;           // [G][J1+1] int (after the warps)
};

template <int D, int G>
__global__ void __launch_bounds__(kRfW * 32) refine8_kernel(const SparseArgs a,
                                                          const __grid_constant__ SeqArgs seq_arg, int round) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  using Lt = RfLayout<D, G>;
  constexpr int CPL = D / 32;          // channels per lane in the query code
  constexpr int CH = D / 16;           // 16-byte chunks per 8-bit row
  constexpr int KS = D / 32;           // k-steps of the dots
  extern __shared__ __align__(16) uint8_t dsm[];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int BG = a.B * a.Hkv;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  const int J = seq.J[b];
  const int JS = a.J1 + 1;
  const int bh0 = b * a.Hq + g * G;
  const int lold = a.front[round * BG + bg] - 1;
  int lnew = -1;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int* st = a.state + (int64_t)(bh0 + h) * 4;
    if (!(st[3] & kFlagDone)) lnew = max(lnew, st[1]);
  }
  if (lnew <= lold) return;
  if (a.refine8 == 2 && round == 0 && lnew < a.r) return;   // a group that stops near level 0
  int* s_hd = reinterpret_cast<int*>(dsm + Lt::hist);
  for (int i = tid; i < G * JS; i += kRfW * 32) s_hd[i] = 0;
  __syncthreads();
  uint8_t* my = dsm + w * Lt::per_warp;
  uint8_t* s_rows = my + Lt::rows;
  int8_t* s_dig = reinterpret_cast<int8_t*>(my + Lt::dig);
  float* s_u8 = reinterpret_cast<float*>(my + Lt::ub8);
  // per head: the scaled query channels of this lane and tree(|qt|)
  const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * G) * D;
  float qt[G][CPL], q1[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float ab[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      qt[h][c] = fmul(__bfloat162float(qp[(int64_t)h * D + lane * CPL + c]), a.rs);
      ab[c] = fabsf(qt[h][c]);
    }
    float s1 = local_tree<CPL>(ab);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) s1 = fadd(s1, __shfl_xor_sync(0xffffffffu, s1, o));
    q1[h] = s1;
  }
  float clo[G], cbv[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { clo[h] = cmax_get(a, bh0 + h, 0); cbv[h] = cmax_get(a, bh0 + h, 2); }
  const float neg_r = -(float)a.r;
  uint16_t* jk = a.jkey + (int64_t)bg * a.pcap;
  const int64_t nblk_p = (P + kBlock - 1) / kBlock;
  const int64_t nwarp = (int64_t)gridDim.x * kRfW;
  for (int64_t blk = (int64_t)blockIdx.x * kRfW + w; blk < nblk_p; blk += nwarp) {
    const int64_t k0 = blk * kBlock;
    // keys of the block to refine in this round
    bool sel[2];
    unsigned jkv[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int64_t key = k0 + lane + 32 * x;
      jkv[x] = key < P ? jk[key] : 0x1FFu;
      const int jm = (int)(jkv[x] & 0x1FFu);
      sel[x] = !(jkv[x] & 0x200u) && jm > lold && jm <= lnew;
    }
    const unsigned m0 = __ballot_sync(0xffffffffu, sel[0]), m1 = __ballot_sync(0xffffffffu, sel[1]);
    if (!(m0 | m1)) continue;
    // stage the selected keys' 8-bit rows (others zero), chunk c of row r
    // at chunk c ^ (r mod CH)
    const uint8_t* src = a.K8 + ((int64_t)bg * a.nblk_max * kBlock + k0) * D;
    for (int c = lane; c < 64 * CH; c += 32) {
      const int r = c / CH, part = c - r * CH;
      const bool ok = ((r < 32 ? m0 >> r : m1 >> (r - 32)) & 1u) != 0u;
      cp_async16(s_rows + r * D + ((part ^ (r & (CH - 1))) << 4), ok ? src + (int64_t)r * D + part * 16 : src, ok);
    }
    cp_async_commit();
    // 12-bit query codes of the block per head, as two s8 digits
    const float* mins = a.bounds + ((int64_t)bg * a.nblk_max + blk) * 2 * D;
    const float* dl8 = a.delta8 + ((int64_t)bg * a.nblk_max + blk) * D;
    float mv[CPL], dv[CPL];
    float kabs = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      mv[c] = mins[lane * CPL + c];
      dv[c] = dl8[lane * CPL + c];
      kabs = fmaxf(kabs, fadd(fabsf(mv[c]), fmul(256.0f, dv[c])));
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) kabs = fmaxf(kabs, __shfl_xor_sync(0xffffffffu, kabs, o));
    float alpha8[G], bhi8[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float av[CPL], tb[CPL], ta[CPL], tp[CPL], tn[CPL];
      float amax = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        av[c] = fmul(qt[h][c], dv[c]);
        amax = fmaxf(amax, fabsf(av[c]));
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      float al = 0.f, inv = 0.f;
      if (amax > 0.f) {
        al = fdiv(amax, 2047.0f);
        inv = fdiv(2047.0f, amax);
      }
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float x = rintf(fmul(av[c], inv));
        x = fminf(fmaxf(x, -2047.0f), 2047.0f);
        const int at = (int)x;
        const float r = fsub(av[c], fmul(al, x));
        tb[c] = fmul(qt[h][c], mv[c]);
        ta[c] = fabsf(av[c]);
        tp[c] = fmaxf(r, 0.0f);
        tn[c] = fmaxf(-r, 0.0f);
        const int hi = (at + 128) >> 8;           // floor((at + 128) / 256), in [-8, 8]
        s_dig[(0 * 8 + h) * D + lane * CPL + c] = (int8_t)(at - 256 * hi);
        s_dig[(1 * 8 + h) * D + lane * CPL + c] = (int8_t)hi;
      }
      float Bq = local_tree<CPL>(tb), A1 = local_tree<CPL>(ta), Rp = local_tree<CPL>(tp), Rn = local_tree<CPL>(tn);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        Bq = fadd(Bq, __shfl_xor_sync(0xffffffffu, Bq, o));
        A1 = fadd(A1, __shfl_xor_sync(0xffffffffu, A1, o));
        Rp = fadd(Rp, __shfl_xor_sync(0xffffffffu, Rp, o));
        Rn = fadd(Rn, __shfl_xor_sync(0xffffffffu, Rn, o));
      }
      const float sk = fmul(A1, 0.5000152587890625f);
      const float hi = fadd(sk, fmul(255.0f, Rp));
      const float lo = fadd(sk, fmul(255.0f, Rn));
      const float mag = fadd(fadd(fmul(q1[h], kabs), hi), lo);
      const float marg = fmul(mag, 6.103515625e-05f);     // 2^-14
      alpha8[h] = al;
      bhi8[h] = fadd(fadd(Bq, hi), marg);
    }
    if (G < 8) {
      // padding heads: zero digits
      for (int i = lane; i < (8 - G) * D; i += 32) {
        s_dig[(0 * 8 + G) * D + i] = 0;
        s_dig[(1 * 8 + G) * D + i] = 0;
      }
    }
    cp_async_wait<0>();
    __syncwarp();
    // exact integer dots: 4 tiles of 16 keys x 8 heads, two digits
    const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      const int r0 = 16 * mt + gq, r1 = r0 + 8;
      int acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        // bytes 32ks + 4tq.. (chunk 2ks) and 32ks + 16 + 4tq.. (chunk 2ks + 1)
        const unsigned a0 = *reinterpret_cast<const unsigned*>(s_rows + r0 * D + (((2 * ks) ^ (r0 & (CH - 1))) << 4) + 4 * tq);
        const unsigned a1 = *reinterpret_cast<const unsigned*>(s_rows + r1 * D + (((2 * ks) ^ (r1 & (CH - 1))) << 4) + 4 * tq);
        const unsigned a2 = *reinterpret_cast<const unsigned*>(s_rows + r0 * D + (((2 * ks + 1) ^ (r0 & (CH - 1))) << 4) + 4 * tq);
        const unsigned a3 = *reinterpret_cast<const unsigned*>(s_rows + r1 * D + (((2 * ks + 1) ^ (r1 & (CH - 1))) << 4) + 4 * tq);
#pragma unroll
        for (int dd = 0; dd < 2; ++dd) {
          const unsigned b0 = *reinterpret_cast<const unsigned*>(s_dig + (dd * 8 + gq) * D + 32 * ks + 4 * tq);
          const unsigned b1 = *reinterpret_cast<const unsigned*>(s_dig + (dd * 8 + gq) * D + 32 * ks + 16 + 4 * tq);
          asm volatile(
              "mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
              "{%0,%1,%2,%3};\n"
              : "+r"(acc[dd][0]), "+r"(acc[dd][1]), "+r"(acc[dd][2]), "+r"(acc[dd][3])
              : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = 2 * tq + (e & 1);
        const int r = (e < 2) ? r0 : r1;
        if (h < G) {
          const int I = acc[1][e] * 256 + acc[0][e];
          s_u8[r * 8 + h] = fadd(fmul(alpha8[h], __int2float_rn(I)), bhi8[h]);
        }
      }
    }
    __syncwarp();
    // refined levels of the selected keys
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      if (!sel[x]) continue;
      const int r = lane + 32 * x;
      const int64_t key = k0 + r;
      const float* up = a.ubar + ((int64_t)bg * a.n_max + key) * G;
      int jm = 0x1FF;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float t = a.per_head ? a.t32[((int64_t)bg * a.pcap + key) * G + h] : a.t32[(int64_t)bg * a.pcap + key];
        const float u4 = up[h];
        const int jb = bound_level(u4, cbv[h], t, neg_r, J);
        if (jb > J || u4 >= clo[h]) continue;          // no candidate, or in the head's exact-max set
        const int jr = bound_level(fminf(u4, s_u8[r * 8 + h]), cbv[h], t, neg_r, J);
        a.jref[((int64_t)bg * a.pcap + key) * G + h] = (uint16_t)jr;
        if (jr != jb) {
          atomicAdd(&s_hd[h * JS + jb], -1);
          atomicAdd(&s_hd[h * JS + jr], 1);
        }
        jm = min(jm, jr);
      }
      jk[key] = (uint16_t)((jkv[x] & 0x400u) | 0x200u | (unsigned)min(jm, 0x1FF));
    }
    __syncwarp();
  }
  __syncthreads();
  for (int i = tid; i < G * (J + 2); i += kRfW * 32) {
    const int h = i / (J + 2), l = i - h * (J + 2);
    const int v = s_hd[h * JS + l];
    if (v) atomicAdd(a.jrd + (int64_t)(bh0 + h) * (a.J1 + 1) + l, v);
  }
}

// ------------------------------------------------------------- candidates

constexpr int kTilesPerCta = kCandSeg / kTile;   // key tiles per CTA of the per-key passes

// Dynamic shared memory of the candidate pass: the staged list, then per
// head the bound-level histogram and the estimated-level histograms.
constexpr int cand_smem(int G, int J1) {
  return kTile * kTilesPerCta * 8 + G * J1 * 8 + G * (J1 + 1) * 4 + G * J1 * 4;
}


// One pass over the pool keys of a group (after the exact maximum):
//  * t_i, the bound level jbar_i per head, the candidate list (jbar <= J;
//    the entry carries the head mask and the smallest jbar over the heads,
//    so that a round rescores only the range it newly needs), the
//    histogram of the first level at which a key's K row is needed;
//  * scores reset to -inf for keys outside the exact-max set: a candidate's
//    score is written when it is rescored, and until then it has no event;
//  * value-free level histograms from an estimated score (exact for the
//    exact-max set, ubar minus the block's half width otherwise; the other
//    keys subsampled one tile in eight): counts of light entries and exits
//    and fixed-point heavy weights per level.  They only size the first
//    gather round.
template <int G>
__global__ void __launch_bounds__(256) cand_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                   int span) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  extern __shared__ __align__(16) uint8_t dsm[];
  const int J1 = a.J1, JS = a.J1 + 1;
  // the CTA's candidates, staged here and written out with one global slot
  // reservation (a per-warp reservation on the group's counter serialises)
  uint2* s_list = reinterpret_cast<uint2*>(dsm);
  // estimated levels: light exits and heavy weights at hl, packed
  // (exits << 40) + weight in 2^-18 fixed point; light entries at jl
  unsigned long long* s_hv = reinterpret_cast<unsigned long long*>(dsm + kTile * kTilesPerCta * 8);  // [G][J1]
  unsigned* s_jr = reinterpret_cast<unsigned*>(s_hv + G * J1);                     // [G][JS]
  int* s_cnt = reinterpret_cast<int*>(s_jr + G * JS);                              // [G][J1]
  __shared__ unsigned s_nc[G];
  __shared__ unsigned s_n, s_gbase;
  const int tid = threadIdx.x, lane = tid & 31;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  const int64_t kbase = (int64_t)blockIdx.x * span;
  if (kbase >= P) return;
  const int64_t kstop = min(P, kbase + span);
  const int J = seq.J[b];
  const float neg_r = -(float)a.r;
  for (int i = tid; i < G * JS; i += 256) s_jr[i] = 0u;
  for (int i = tid; i < G * J1; i += 256) { s_cnt[i] = 0; s_hv[i] = 0ull; }
  if (tid < G) s_nc[tid] = 0u;
  if (tid == 0) s_n = 0u;
  __syncthreads();
  const int bh0 = b * a.Hq + g * G;
  float c_lo[G], c_b[G], c32[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    c_lo[h] = cmax_get(a, bh0 + h, 0);
    c_b[h] = cmax_get(a, bh0 + h, 2);
    c32[h] = cmax_get(a, bh0 + h, 3);
  }
  // perturbation keys: the group's, or one per query head
  unsigned long long gk[G];
#pragma unroll
  for (int h = 0; h < G; ++h) gk[h] = group_key(seq.seed[b], a.per_head ? kHeadStream + g * G + h : g);
  const bool inset_all = (int64_t)a.xcnt[bg] * 32 <= P;
  // ubar and the block half widths of a key, loaded one tile ahead
  auto load_key = [&](int64_t k, float (&u)[G], float (&h)[G]) {
    if (k >= P) return;
    const float* up = a.ubar + ((int64_t)bg * a.n_max + k) * G;
    const float* hp = a.hw + ((int64_t)bg * a.nblk_max + k / kBlock) * G;
    if (G == 4) {
      const float4 f = *reinterpret_cast<const float4*>(up);
      u[0] = f.x; u[1 % G] = f.y; u[2 % G] = f.z; u[3 % G] = f.w;
      const float4 e = *reinterpret_cast<const float4*>(hp);
      h[0] = e.x; h[1 % G] = e.y; h[2 % G] = e.z; h[3 % G] = e.w;
    } else {
#pragma unroll
      for (int x = 0; x < G; ++x) { u[x] = up[x]; h[x] = hp[x]; }
    }
  };
  float ub[G], hw[G], nub[G], nhw[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { ub[h] = hw[h] = nub[h] = nhw[h] = 0.f; }
  load_key(kbase + tid, ub, hw);
  int tile = 0;
  for (int64_t key0 = kbase; key0 < kstop; key0 += kTile, ++tile) {
  const int64_t key = key0 + tid;
  const bool live = key < kstop;
  if (key0 + kTile < kstop) load_key(key + kTile, nub, nhw);
  unsigned cm = 0;
  bool inset = false;
  float t[G];
#pragma unroll
  for (int h = 0; h < G; ++h) t[h] = 0.f;
  if (live) {
    if (a.per_head) {
#pragma unroll
      for (int h = 0; h < G; ++h) t[h] = perturb_t(gk[h], key);
      float* tp = a.t32 + ((int64_t)bg * a.pcap + key) * G;
      if (G == 4) *reinterpret_cast<float4*>(tp) = make_float4(t[0], t[1 % G], t[2 % G], t[3 % G]);
      else {
#pragma unroll
        for (int h = 0; h < G; ++h) tp[h] = t[h];
      }
    } else {
      const float t0 = perturb_t(gk[0], key);
#pragma unroll
      for (int h = 0; h < G; ++h) t[h] = t0;
      a.t32[(int64_t)bg * a.pcap + key] = t0;
    }
  }
  int jmin = 255, jmin_out = 0x1FF;   // jmin_out: over the heads not in their exact-max set
#pragma unroll
  for (int h = 0; h < G; ++h) {
    bool inc = false;
    if (live) {
      const int jb = bound_level(ub[h], c_b[h], t[h], neg_r, J);
      const bool cand = jb <= J;
      inc = ub[h] >= c_lo[h];
      inset |= inc;
      if (cand) { cm |= 1u << h; jmin = min(jmin, jb); }
      if (cand && !inc) jmin_out = min(jmin_out, jb);
      // first level the row is needed (keys never needed are not counted:
      // most keys of a peaked group, all on one shared-memory word)
      if (inc || cand) atomicAdd(&s_jr[h * JS + (inc ? 0 : jb)], 1u);
    }
    const unsigned cb = __ballot_sync(0xffffffffu, (cm >> h) & 1u);
    if (lane == 0 && cb) atomicAdd(&s_nc[h], (unsigned)__popc(cb));
    if (a.refine8) {
      const unsigned ib = __ballot_sync(0xffffffffu, inc);
      if (lane == 0 && ib) atomicAdd(a.ninset + bh0 + h, (unsigned)__popc(ib));
    }
  }
  if (a.refine8 && live)
    a.jkey[(int64_t)bg * a.pcap + key] = (uint16_t)(inset ? (0x400u | (unsigned)jmin_out) : (unsigned)jmin_out);
  float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
  // estimated levels (a key that is no candidate of a head has no level
  // up to J for it): one tile in eight with weight 8; when the exact-max
  // set is small (it then holds the few keys that carry the heavy weight)
  // its keys on every tile with weight 1.  (One tile in 4, 8, 16: 717,
  // 709, 715 us per 128K x 4 step; sparser samples blur the prediction.)
  const bool samp = (tile & 7) == 0;
  if (samp || (inset_all && __any_sync(0xffffffffu, live && inset))) {
    const unsigned mult = (live && inset && inset_all) ? 1u : (live && samp ? 8u : 0u);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      int jl = J + 1, hl = J + 1;
      float est = 0.f;
      if (mult && ((cm >> h) & 1u)) {
        est = inset ? sp[h] : fsub(ub[h], hw[h]);
        exact_levels(est, c32[h], t[h], neg_r, J, jl, hl);
      }
      // plain per-lane shared atomics (aggregating over equal levels first
      // cost more than the conflicts it saved)
      if (jl < hl) atomicAdd(&s_cnt[h * J1 + jl], (int)mult);                        // light from jl
      if (hl <= J)                                                                   // light until hl,
        atomicAdd(&s_hv[h * J1 + hl], ((unsigned long long)(jl < hl ? mult : 0u) << 40) +   // heavy from hl
                                          mult * __float2uint_rn(__expf(fminf(est - c32[h], 0.f)) * 262144.f));
    }
  }
  if (live && inset) {
    // scored in the exact-max step: keep the candidate heads' scores
#pragma unroll
    for (int h = 0; h < G; ++h)
      if (!((cm >> h) & 1u)) sp[h] = -INFINITY;
  } else if (live) {
#pragma unroll
    for (int h = 0; h < G; ++h) sp[h] = -INFINITY;
  }
  const int slot = warp_append(&s_n, live && !inset && cm);
  if (slot >= 0) s_list[slot] = make_uint2((unsigned)key, cm | ((unsigned)jmin << 8));
#pragma unroll
  for (int h = 0; h < G; ++h) { ub[h] = nub[h]; hw[h] = nhw[h]; }
  if ((tile + 1) % kTilesPerCta == 0 || key0 + kTile >= kstop) {
    __syncthreads();
    if (tid == 0) s_gbase = s_n ? atomicAdd(a.ccnt + bg, s_n) : 0u;
    __syncthreads();
    for (unsigned i = tid; i < s_n; i += 256) a.clist[(int64_t)bg * a.pcap + s_gbase + i] = s_list[i];
    __syncthreads();
    if (tid == 0) s_n = 0u;
    __syncthreads();
  }
  }
  __syncthreads();
  for (int i = tid; i < G * (J + 2); i += 256) {
    int h = i / (J + 2), l = i - h * (J + 2);
    unsigned v = s_jr[h * JS + l];
    if (v) atomicAdd(a.jr_hist + (int64_t)(bh0 + h) * (a.J1 + 1) + l, v);
  }
  if (tid < G && s_nc[tid]) atomicAdd(a.ncand + bh0 + tid, s_nc[tid]);
  for (int i = tid; i < G * (J + 1); i += 256) {
    const int h = i / (J + 1), l = i - h * (J + 1);
    float* dst = a.pre_hist + ((int64_t)(bh0 + h) * a.J1 + l) * 4;
    const unsigned long long hv = s_hv[h * J1 + l];
    const int dk = s_cnt[h * J1 + l] - (int)(hv >> 40);
    const unsigned long long db = hv & ((1ull << 40) - 1ull);
    if (dk) atomicAdd(dst + 0, (float)dk);
    if (db) atomicAdd(dst + 1, (float)db * 3.814697265625e-06f);   // 2^-18
  }
}

// -------------------------------------------- window sums + stop predictor

template <int D, int G, typename E>
__global__ void __launch_bounds__(256) predict_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  constexpr int CPL = D / 32;
  __shared__ float s_nr[G][D];
  __shared__ float s_dr[G], s_hr[G];
  __shared__ float s_vm[8];
  __shared__ float s_wp[8][G][D + 2];     // per-warp window partials
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bg = blockIdx.x, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  const int bh0 = b * a.Hq + g * G;
  if (n <= kWindow) {
    // no pool: dense attention for every head of the group
    if (tid < G) {
      int* st = a.state + (int64_t)(bh0 + tid) * 4;
      st[0] = 0; st[1] = 0; st[2] = 0; st[3] = kFlagFallback | kFlagDone;
      atomicAdd(a.nfall, 1u);
    }
    return;
  }
  const int64_t P = n - kWindow;
  const int J = seq.J[b];
  for (int i = tid; i < G * D; i += 256) (&s_nr[0][0])[i] = 0.f;
  if (tid < G) { s_dr[tid] = 0.f; s_hr[tid] = 0.f; }
  __syncthreads();
  // every load of this phase is issued before its values are used: the
  // warp's eight window rows and their scores, c32, and (below) the pool's
  // value-norm bounds
  constexpr int RPW = kWindow / 8;   // window rows per warp
  const E* Vb = reinterpret_cast<const E*>(a.V) + ((int64_t)bg * a.n_max + P) * D;
  float vw[RPW][CPL], sw[RPW][G];
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int row = w + 8 * i;
    load_row<D, E>(Vb + (int64_t)row * D, vw[i]);
    const float* ws = a.win + ((int64_t)bg * kWindow + row) * G;
#pragma unroll
    for (int h = 0; h < G; ++h) sw[i][h] = ws[h];
  }
  float c32[G];
#pragma unroll
  for (int h = 0; h < G; ++h) c32[h] = cmax_get(a, bh0 + h, 3);
  float vmx = 0.f;
  {
    const int64_t nbp = (P + kBlock - 1) / kBlock;
#pragma unroll 8
    for (int64_t i = tid; i < nbp; i += 256) vmx = fmaxf(vmx, a.vmax[(int64_t)bg * a.nblk_max + i]);
  }
  float nr[G][CPL], dr[G], hr[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    dr[h] = 0.f; hr[h] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) nr[h][c] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    float sq = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) sq += vw[i][c] * vw[i][c];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float wt = expf(fsub(sw[i][h], c32[h]));
      dr[h] += wt;
      hr[h] += wt * sq;
#pragma unroll
      for (int c = 0; c < CPL; ++c) nr[h][c] += wt * vw[i][c];
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) s_wp[w][h][lane * CPL + c] = nr[h][c];
    const float hs = warp_sum(hr[h]);       // lanes hold channel partials
    if (lane == 0) { s_wp[w][h][D] = dr[h]; s_wp[w][h][D + 1] = hs; }   // dr: same in every lane
  }
  // largest value-norm bound over the pool blocks
  {
    const float m = warp_max(vmx);
    if (lane == 0) s_vm[w] = m;
  }
  __syncthreads();
  // window sums: the eight warps' partials in a fixed order
  for (int i = tid; i < G * (D + 2); i += 256) {
    const int h = i / (D + 2), c = i - h * (D + 2);
    float v = 0.f;
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) v += s_wp[ww][h][c];
    if (c < D) s_nr[h][c] = v;
    else if (c == D) s_dr[h] = v;
    else s_hr[h] = v;
  }
  __syncthreads();
  float Vp = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) Vp = fmaxf(Vp, s_vm[i]);
  if (tid == 0) a.vmaxp[bg] = Vp;
  for (int i = tid; i < G * (D + 4); i += 256) {
    int h = i / (D + 4), c = i - h * (D + 4);
    float v = c < D ? s_nr[h][c] : (c == D ? s_dr[h] : (c == D + 1 ? s_hr[h] : 0.f));
    a.winstats[(int64_t)(bh0 + h) * (D + 4) + c] = v;
  }
  // value-free stop prediction: warp h, lanes over levels
  if (w < G) {
    const int h = w, bh = bh0 + h;
    const float DR = s_dr[h], HR = s_hr[h];
    float cn2 = 0.f;
    for (int c = lane; c < D; c += 32) { float x = s_nr[h][c] / DR; cn2 += x * x; }
    cn2 = warp_sum(cn2);
    const float nu = HR / DR;
    const float cn = sqrtf(cn2);
    const float de = a.delta / (4.0f * (float)(J + 1));
    const float L = logf(1.0f / de), Lz = logf(2.0f / de);
    const float Rc = Vp + cn;
    // pred: first level the value-free certificate passes; round 1 gathers
    // max(1, r - 1) levels past it (the estimate tends to pass a few levels
    // early on peaked heads; margins of 1, 2, 3 and 4 levels at r = 4 gave
    // 763, 722, 716 and 719 us per 128K x 4 step)
    float runk = 0.f, rundb = 0.f;
    int pred = -1;
    // the histogram of a chunk of 32 levels, loaded one chunk ahead
    auto load_chunk = [&](int l0, float& dk, float& ddb) {
      dk = 0.f; ddb = 0.f;
      if (l0 + lane <= J) {
        const float* ph = a.pre_hist + ((int64_t)bh * a.J1 + l0 + lane) * 4;
        dk = ph[0]; ddb = ph[1];
      }
    };
    float nk, ndb;
    load_chunk(0, nk, ndb);
    for (int l0 = 0; l0 <= J; l0 += 32) {
      const int j = l0 + lane;
      const float dk = nk, ddb = ndb;
      load_chunk(l0 + 32, nk, ndb);
      // inclusive scan over the 32 lanes
      float k = dk, db = ddb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        float x = __shfl_up_sync(0xffffffffu, k, o), y = __shfl_up_sync(0xffffffffu, db, o);
        if (lane >= o) { k += x; db += y; }
      }
      k += runk; db += rundb;
      runk = __shfl_sync(0xffffffffu, k, 31);
      rundb = __shfl_sync(0xffffffffu, db, 31);
      bool pass = false;
      if (j <= J) {
        const float tau = exp2f(-(float)j / (float)a.r);
        float below, above;
        chernoff_gaps(k, Lz, below, above);
        const float dD = tau * fmaxf(below, above);
        const float Dh = DR + db + tau * k;
        if (a.measure == CSA_MEASURE_DENOM) {
          pass = Dh > dD && dD <= a.eps * (Dh - dD);
        } else if (a.measure == CSA_MEASURE_CLT) {
          const float Gh = tau * k * fmaxf(nu - cn2, 0.f);
          const float Mh = sqrtf((HR + db * nu + tau * k * nu) / Dh);
          pass = Dh > 0.f && a.zclt * sqrtf(tau * Gh) <= a.eps * Mh * Dh;
        } else {
          const float Gh = tau * k * fmaxf(nu - cn2, 0.f);
          const float aa = sqrtf(2.f * tau * Rc * Rc * L);
          const float sq = sqrtf(aa * aa + 4.f * (Gh + (2.f / 3.f) * tau * Rc * Rc * L));
          const float Ghi = 0.25f * (aa + sq) * (aa + sq);
          const float zeta = sqrtf(2.f * tau * Ghi * Lz) + (2.f / 3.f) * tau * Rc * Lz;
          const float beta = Dh > dD ? zeta / (Dh - dD) : INFINITY;
          float scale;
          if (a.measure == CSA_MEASURE_VALUE) {
            const float Hh = tau * k * nu;
            const float ap = sqrtf(2.f * tau * Vp * Vp * L);
            const float br = Hh - (2.f / 3.f) * tau * Vp * Vp * L;
            const float t2 = br > 0.f ? 0.5f * (-ap + sqrtf(ap * ap + 4.f * br)) : 0.f;
            const float Mlo = sqrtf((HR + db * nu + t2 * t2) / (DR + db + tau * (k + above)));
            scale = Mlo;
            pass = Dh > dD && beta <= a.eps * scale;
          } else {
            pass = Dh > dD && beta * (1.f + a.eps) <= a.eps * cn;
          }
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, pass);
      if (bal) { pred = l0 + __ffs(bal) - 1; break; }
    }
    if (lane == 0) {
      // (a prediction of level 0, the flat heads', is not widened: it was
      // exact on every flat head measured, and level 1 would add ~20% rows)
      const int margin = a.r > 2 ? a.r - 1 : 1;
      const int hi = pred < 0 ? J : (pred == 0 ? 0 : min(J, pred + margin));
      int* st = a.state + (int64_t)bh * 4;
      st[0] = -1; st[1] = hi; st[2] = -1; st[3] = 0;
    }
  }
  if (tid == 0) rq_push(a, 0, bg);
}

// --------------------------------------------------------- level buckets

#ifndef CSA_LEV_ITEM
#define CSA_LEV_ITEM 2048
#endif
constexpr int kLevItem = CSA_LEV_ITEM;   // keys per work item of the level pass (first round)
constexpr int kLevItemLate = 512; // later rounds: few groups, more and shorter items
#ifndef CSA_LEV_CPS
#define CSA_LEV_CPS 8
#endif
constexpr int kLevCps = CSA_LEV_CPS;   // level-pass CTAs launched per SM (at most)

// One work item: keys [k0, k0 + isz) of group bg.
template <int G, bool PH>
__device__ __forceinline__ void levels_item(const SparseArgs& a, const SeqArgs& seq, int bg, int64_t k0,
                                            int isz, int round, uint2* sev) {
  const int lane = threadIdx.x & 31;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  if (k0 >= P) return;
  const int64_t kend = min(P, k0 + isz);
  const int J = seq.J[b];
  const int bh0 = b * a.Hq + g * G;
  const float* sb = a.s32 + (int64_t)bg * a.pcap * G;
  const float* tb = a.t32 + (int64_t)bg * a.pcap * (PH ? G : 1);
  // scores and t of a key, loaded one 256-key step ahead
  auto load_key = [&](int64_t k, float (&sv)[G], float (&t)[G]) {
#pragma unroll
    for (int h = 0; h < G; ++h) { sv[h] = -INFINITY; t[h] = 0.f; }
    if (k >= kend) return;
    if (G == 4) {
      const float4 f = *reinterpret_cast<const float4*>(sb + k * G);
      sv[0] = f.x; sv[1 % G] = f.y; sv[2 % G] = f.z; sv[3 % G] = f.w;
    } else {
#pragma unroll
      for (int h = 0; h < G; ++h) sv[h] = sb[k * G + h];
    }
    if (PH) {
#pragma unroll
      for (int h = 0; h < G; ++h) t[h] = tb[k * G + h];
    } else {
      const float t0 = tb[k];
#pragma unroll
      for (int h = 0; h < G; ++h) t[h] = t0;
    }
  };
  // the item's first keys, c32 and the heads' ranges load together (one
  // round trip before the first tile, not three)
  float cs[G], ns[G], ct[G], nt[G];
  load_key(k0 + threadIdx.x, cs, ct);
  float c32[G];
#pragma unroll
  for (int h = 0; h < G; ++h) c32[h] = cmax_get(a, bh0 + h, 3);
  int lo[G], hi[G];
  int whi = -1;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int* st = a.state + (int64_t)(bh0 + h) * 4;
    lo[h] = st[0];
    hi[h] = (st[3] & kFlagDone) ? st[0] : st[1];
    if (hi[h] > lo[h]) whi = max(whi, hi[h]);
  }
  if (whi < 0) return;
  const float neg_r = -(float)a.r;
  // this round's bucket counters (one set per round, zeroed with the step)
  unsigned* bcnt = a.bcnt + ((int64_t)round * a.B * a.Hkv + bg) * a.J1;
  uint2* bk = a.buckets + (int64_t)bg * a.J1 * a.pcap;
  for (int64_t key0 = k0; key0 < kend; key0 += 256) {
    const int64_t key = key0 + threadIdx.x;
    load_key(key + 256, ns, nt);
    int jl[G], hl[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      jl[h] = J + 1; hl[h] = J + 1;
      if (cs[h] > -INFINITY) exact_levels(cs[h], c32[h], ct[h], neg_r, J, jl[h], hl[h]);
      cs[h] = ns[h];
      ct[h] = nt[h];
    }
    // the key's entries for the round's levels: for each head a light
    // entry at jl < hl in its range (bit h) and the move to the heavy sums
    // at hl in its range (bit 8 + h, and bit 16 + h when the key was light
    // before), one entry per distinct level with every head's bits merged
    // (a bucket holds at most one entry per key in a round).  The warp
    // first packs its lanes' entries into shared memory (the level in bits
    // 24-31 of the mask word), then takes them 32 at a time: lanes with the
    // same level share one slot reservation, so a warp makes one round trip
    // to the counters per 32 entries rather than one per level of a lane.
    unsigned pa = 0, pt = 0;
    if (key < kend) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (jl[h] < hl[h] && jl[h] > lo[h] && jl[h] <= hi[h]) pa |= 1u << h;
        if (hl[h] <= J && hl[h] > lo[h] && hl[h] <= hi[h]) pt |= 1u << h;
      }
    }
    unsigned nev = 0;
#pragma unroll
    for (int k = 0; k < 2 * G; ++k) {
      if (!__any_sync(0xffffffffu, (pa | pt) != 0u)) break;
      int cur = 1 << 20;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if ((pa >> h) & 1u) cur = min(cur, jl[h]);
        if ((pt >> h) & 1u) cur = min(cur, hl[h]);
      }
      unsigned m = 0;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (((pa >> h) & 1u) && jl[h] == cur) { m |= 1u << h; pa &= ~(1u << h); }
        if (((pt >> h) & 1u) && hl[h] == cur) {
          m |= 1u << (8 + h);
          if (jl[h] < hl[h]) m |= 1u << (16 + h);
          pt &= ~(1u << h);
        }
      }
      const unsigned bal = __ballot_sync(0xffffffffu, m != 0u);
      if (m) sev[nev + __popc(bal & ((1u << lane) - 1u))] = make_uint2((unsigned)key, m | ((unsigned)cur << 24));
      nev += __popc(bal);
    }
    __syncwarp();
    for (unsigned i0 = 0; i0 < nev; i0 += 32) {
      const bool has = i0 + lane < nev;
      const uint2 e = has ? sev[i0 + lane] : make_uint2(0u, 0u);
      const int l = has ? (int)(e.y >> 24) : -1;
      const unsigned grp = __match_any_sync(0xffffffffu, l);
      const int leader = __ffs(grp) - 1;
      unsigned p0 = 0;
      if (lane == leader && l >= 0) p0 = atomicAdd(bcnt + l, (unsigned)__popc(grp));
      p0 = __shfl_sync(0xffffffffu, p0, leader);
      if (l >= 0) {
        const unsigned p = p0 + (unsigned)__popc(grp & ((1u << lane) - 1u));
        if (p < (unsigned)a.pcap) bk[(int64_t)l * a.pcap + p] = make_uint2(e.x, e.y & 0x00FFFFFFu);
        else atomicOr(a.status, 2u);
      }
    }
    __syncwarp();
  }
}

template <int G, bool PH>
__global__ void __launch_bounds__(256) levels_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                     int round, unsigned tpg, int isz) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  __shared__ unsigned s_item;
  __shared__ uint2 s_ev[8][64 * G];      // per warp: up to 2G entries per lane
  const int BG = a.B * a.Hkv;
  const unsigned total = a.rq[6 * BG + round] * tpg;
  for (;;) {
    if (threadIdx.x == 0) s_item = atomicAdd(a.rq + 6 * BG + 3 + round, 1u);
    __syncthreads();
    const unsigned item = s_item;
    __syncthreads();
    if (item >= total) break;
    levels_item<G, PH>(a, seq, (int)a.rq[round * BG + item / tpg], (int64_t)(item % tpg) * isz, isz, round,
                       s_ev[threadIdx.x >> 5]);
  }
}

// One CTA: the bucket entries appended in this round, as per-bucket ranges
// [plan_start, plan_end) and their exclusive prefix plan_off over the
// buckets.  EV: the prefix counts work units, the entries plus
// kVsBucketCost per non-empty bucket (the tensor-core gather cuts it into
// equal per-warp ranges); otherwise it counts work items of kChunk entries
// and chunk_map maps each item to its bucket.
template <bool EV>
__global__ void __launch_bounds__(1024) vplan_kernel(const SparseArgs a, int nent, int round) {
  pdl_entry();
  __shared__ unsigned s_part[1024];
  const int tid = threadIdx.x;
  const int per = (nent + 1023) / 1024;
  const int i0 = tid * per, i1 = min(nent, i0 + per);
  unsigned sum = 0;
  const unsigned* cnt = a.bcnt + (int64_t)round * nent;   // this round's counters
  for (int i = i0; i < i1; ++i) {
    // this round's entries (a bucket holds at most one entry per key in a
    // round); the step's cumulative count is kept in bcons (diagnostics)
    const unsigned st = 0;
    unsigned en = cnt[i];
    if (en > (unsigned)a.pcap) en = (unsigned)a.pcap;
    a.plan_start[i] = st;
    a.plan_end[i] = en;
    a.bcons[i] += en;
    sum += EV ? en - st + (en > st ? kVsBucketCost : 0u) : (en - st + kChunk - 1) / kChunk;
  }
  // exclusive prefix of the per-thread sums: a shuffle scan within each
  // warp, then one over the 32 warp totals
  const int lane = tid & 31, wp = tid >> 5;
  unsigned inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned x = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += x;
  }
  if (lane == 31) s_part[wp] = inc;
  __syncthreads();
  if (wp == 0) {
    unsigned t = s_part[lane], ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned x = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += x;
    }
    s_part[32 + lane] = ti - t;          // exclusive warp offsets
    if (lane == 31) s_part[64] = ti;     // total
  }
  __syncthreads();
  unsigned run = s_part[32 + wp] + inc - sum;
  for (int i = i0; i < i1; ++i) {
    a.plan_off[i] = run;
    if (EV) {
      const unsigned ne = a.plan_end[i] - a.plan_start[i];
      run += ne + (ne ? kVsBucketCost : 0u);
    } else {
      const unsigned nch = (a.plan_end[i] - a.plan_start[i] + kChunk - 1) / kChunk;
      for (unsigned k = 0; k < nch; ++k)
        if (run + k < (unsigned)a.nchunk_cap) a.chunk_map[run + k] = (unsigned)i;
      run += nch;
    }
  }
  if (tid == 1023) {
    unsigned tot = s_part[64];
    a.plan_off[nent] = (EV || tot < (unsigned)a.nchunk_cap) ? tot : (unsigned)a.nchunk_cap;
  }
}

// ------------------------------------------------------------- V gather

constexpr int kVgW = 8;   // warps per CTA of the float32 value gather (256 threads)
constexpr int kVgS = 4;   // its ring stages per warp (8 rows each)

template <int D, int G, typename E>
constexpr int vgather_smem() {
  return kVgW * kVgS * 8 * D * (int)sizeof(E) + kVgW * kVgS * 8 * 16 + G * (2 * D + 8) * 4 +
         kVgW * (kChunk / kVgW) * 8 + kVgW * kVgS * 8 * G * 4;
}

template <int D, int G, typename E>
__global__ void __launch_bounds__(256) vgather_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                      int nent) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  constexpr int CPL = D / 32;
  constexpr int ACC = 2 * D + 8;
  constexpr int RB = D * (int)sizeof(E);
  constexpr int EPW = kChunk / kVgW;          // events per warp per work item
  extern __shared__ __align__(16) uint8_t dsm[];
  uint8_t* ring = dsm;
  float* s_sc = reinterpret_cast<float*>(dsm + kVgW * kVgS * 8 * RB);            // [W][S][8][4]
  float (*s_acc)[ACC] = reinterpret_cast<float (*)[ACC]>(dsm + kVgW * kVgS * 8 * RB + kVgW * kVgS * 8 * 16);
  uint2* s_ev = reinterpret_cast<uint2*>(dsm + kVgW * kVgS * 8 * RB + kVgW * kVgS * 8 * 16 + G * ACC * 4);
  float* s_ww = reinterpret_cast<float*>(dsm + kVgW * kVgS * 8 * RB + kVgW * kVgS * 8 * 16 + G * ACC * 4 +
                                         kVgW * EPW * 8);                       // [W][S][8][G]
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const unsigned total = a.plan_off[nent];
  uint8_t* my = ring + w * kVgS * 8 * RB;
  float* msc = s_sc + w * kVgS * 8 * 4;
  uint2* mev = s_ev + w * EPW;
  float* mww = s_ww + w * kVgS * 8 * G;
  for (unsigned c = blockIdx.x; c < total; c += gridDim.x) {
    const int e = (int)a.chunk_map[c];
    const int bg = e / a.J1, l = e - bg * a.J1;
    const int b = bg / a.Hkv, g = bg - b * a.Hkv;
    const int bh0 = b * a.Hq + g * G;
    const unsigned ev0 = a.plan_start[e] + (c - a.plan_off[e]) * kChunk;
    const unsigned ev1 = min(a.plan_end[e], ev0 + kChunk);
    // this warp's batches of eight events: w, w + 8, w + 16, ... of the
    // work item (balanced over the warps), loaded in one sweep
    const int nev = (int)(ev1 - ev0);
    const int nball = (nev + 7) / 8;
    const int nmy = nball > w ? (nball - w + kVgW - 1) / kVgW : 0;   // batches of this warp
    const uint2* bk = a.buckets + (int64_t)e * a.pcap + ev0;
#pragma unroll
    for (int i = lane; i < EPW; i += 32) {
      const int k = i >> 3, r = i & 7;
      const int idx = (w + k * kVgW) * 8 + r;
      mev[i] = (k < nmy && idx < nev) ? bk[idx] : make_uint2(0u, 0u);
    }
    float c32[G];
#pragma unroll
    for (int h = 0; h < G; ++h) c32[h] = cmax_get(a, bh0 + h, 3);
    __syncthreads();
    for (int i = tid; i < G * ACC; i += 256) (&s_acc[0][0])[i] = 0.f;
    __syncthreads();
    float S1[G][CPL], NB[G][CPL], s2[G], hb[G], kc[G], db[G], ns[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      s2[h] = hb[h] = kc[h] = db[h] = ns[h] = 0.f;
#pragma unroll
      for (int x = 0; x < CPL; ++x) { S1[h][x] = 0.f; NB[h][x] = 0.f; }
    }
    unsigned hm = 0;
    const E* Vb = reinterpret_cast<const E*>(a.V) + (int64_t)bg * a.n_max * D;
    const float* sb = a.s32 + (int64_t)bg * a.pcap * G;
    const int nbatch = nmy;
    // events in the warp's k-th batch
    auto bcount = [&](int k) { return k < nmy ? min(8, nev - (w + k * kVgW) * 8) : 0; };
    auto issue = [&](int slot, int bt) {
      const int nv = bcount(bt);
      stage8<D, E>(my + slot * 8 * RB, Vb, mev + bt * 8, nv);
      // the G scores of each event (16-byte rows of s32 when G = 4)
      if (lane < 8) {
        const bool ok = lane < nv;
        const float* src = ok ? sb + (int64_t)mev[bt * 8 + lane].x * G : sb;
        if (G == 4) cp_async16(msc + (slot * 8 + lane) * 4, src, ok);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int sl = 0; sl < kVgS; ++sl) issue(sl, sl);
    for (int bt = 0; bt < nbatch; ++bt) {
      const int slot = bt & (kVgS - 1);
      cp_async_wait<kVgS - 1>();
      __syncwarp();
      const int nv = bcount(bt);
      // transition weights, one lane per event
      if (lane < nv) {
        const uint2 ev = mev[bt * 8 + lane];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float ww = 0.f;
          if (ev.y & (1u << (8 + h))) {
            const float sh = G == 4 ? msc[(slot * 8 + lane) * 4 + h] : sb[(int64_t)ev.x * G + h];
            ww = expf(fsub(sh, c32[h]));
          }
          mww[(slot * 8 + lane) * G + h] = ww;
        }
      }
      __syncwarp();
      for (int r = 0; r < nv; ++r) {
        const uint2 ev = mev[bt * 8 + r];
        const unsigned m = ev.y;
        hm |= m;
        float v[CPL];
        load_row<D, E>(reinterpret_cast<const E*>(my + (slot * 8 + r) * RB), v);
        float sq = 0.f;
#pragma unroll
        for (int x = 0; x < CPL; ++x) sq += v[x] * v[x];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const bool add = m & (1u << h), trn = m & (1u << (8 + h)), bef = m & (1u << (16 + h));
          if (add) {
#pragma unroll
            for (int x = 0; x < CPL; ++x) S1[h][x] += v[x];
            s2[h] += sq;
            kc[h] += 1.f;
            ns[h] += 1.f;
          }
          if (trn) {
            const float ww = mww[(slot * 8 + r) * G + h];
            if (bef) {
#pragma unroll
              for (int x = 0; x < CPL; ++x) S1[h][x] -= v[x];
              s2[h] -= sq;
              kc[h] -= 1.f;
            } else {
              ns[h] += 1.f;
            }
#pragma unroll
            for (int x = 0; x < CPL; ++x) NB[h][x] += ww * v[x];
            hb[h] += ww * sq;
            db[h] += ww;
          }
        }
      }
      __syncwarp();
      issue(slot, bt + kVgS);
    }
    cp_async_wait<0>();
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (!(hm & (0x101u << h))) continue;
#pragma unroll
      for (int x = 0; x < CPL; ++x) {
        atomicAdd(&s_acc[h][lane * CPL + x], S1[h][x]);
        atomicAdd(&s_acc[h][D + lane * CPL + x], NB[h][x]);
      }
      const float s2_ = warp_sum(s2[h]), hb_ = warp_sum(hb[h]);
      if (lane == 0) {
        // counts and weights are the same in every lane
        atomicAdd(&s_acc[h][2 * D + 0], kc[h]);
        atomicAdd(&s_acc[h][2 * D + 1], s2_);
        atomicAdd(&s_acc[h][2 * D + 2], db[h]);
        atomicAdd(&s_acc[h][2 * D + 3], hb_);
        atomicAdd(&s_acc[h][2 * D + 4], ns[h]);
      }
    }
    __syncthreads();
    for (int i = tid; i < G * ACC; i += 256) {
      const int h = i / ACC, x = i - h * ACC;
      if (x >= 2 * D + 5) continue;
      const float v = s_acc[h][x];
      if (v != 0.f) atomicAdd(a.acc + ((int64_t)(bh0 + h) * a.J1 + l) * ACC + x, v);
    }
  }
}

// Tensor-core V gather (bf16 caches).  The round's new bucket entries,
// concatenated bucket after bucket, are cut into one contiguous range per
// warp.  A warp walks its range in batches of 16 entries of one bucket
// (one level of one group), staging the 16 value rows, the candidates'
// scores and their ||v||^2 in a per-warp ring filled with cp.async, and
// accumulates
//   C += A Vx,   Vx = [value rows | 1, hi(||v||^2), lo(||v||^2), 0...]
// where A has 4G rows per event column: rows 0..G-1 the light coefficient
// (+1 on a light entry, -1 when a light key turns heavy), rows G..2G-1 and
// 2G..3G-1 the heavy weight w = exp(s - c32) split as bf16(w) and
// bf16(w - bf16(w)) so the product stays float32-accurate, rows 3G..4G-1
// the sampled-key flag.  One batch is (D/8 + 1) mma per 16 rows of A.  The
// accumulators go to the per-level sums with vector reductions whenever the
// bucket changes and at the end of the range.
#ifndef CSA_VS_WARPS
#define CSA_VS_WARPS 4
#endif
#ifndef CSA_VS_STAGES
#define CSA_VS_STAGES 4
#endif
// (stages x warps on the 128K x 4 step, two chains: 3 x 4 623-627 us,
// 4 x 4 620-621, 2 x 8 623-624, 2 x 4 625-628, 3 x 2 635-638)
constexpr int kVsW = CSA_VS_WARPS;              // warps per CTA
constexpr int kVsS = CSA_VS_STAGES;             // row stages per warp (>= 2)
constexpr int kVsE = 2 * kVsS;                  // entry / descriptor slots per warp
constexpr int kVsB = 16;                        // entries per batch (mma k)

template <int D, int G>
struct VsLayout {
  static constexpr int RB = 2 * D;                               // bf16 value row
  static constexpr int MT = (4 * G + 15) / 16;                   // m-tiles of A
  static constexpr int SCB = 4 * G;                              // scores per entry
  static constexpr int rows = 0;
  static constexpr int sc = rows + kVsS * kVsB * RB;
  static constexpr int vn = sc + kVsS * kVsB * SCB;
  static constexpr int ent = vn + kVsS * kVsB * 4;
  static constexpr int desc = ent + kVsE * kVsB * 8;             // [e, entry offset, count, bg, c32 x 8]
  static constexpr int atb = kVsB * MT * 32;                     // A^T: [16 entries][16 MT] bf16
  static constexpr int at = desc + kVsE * 64;                    // two A^T buffers
  static constexpr int bx = at + 2 * atb;                        // two [16 entries][8] bf16
  static constexpr int per_warp = bx + 2 * kVsB * 16;
  static constexpr int smem = kVsW * per_warp;
};

template <int BYTES>
__device__ __forceinline__ void cp_async_small(void* smem, const void* gmem, bool valid) {
  unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  int src = valid ? BYTES : 0;
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;\n" ::"r"(sa), "l"(gmem), "n"(BYTES), "r"(src));
}

__device__ __forceinline__ void ldsm_x4_trans(unsigned (&r)[4], const void* p) {
  unsigned sa = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(sa));
}
__device__ __forceinline__ void ldsm_x2_trans(unsigned (&r)[2], const void* p) {
  unsigned sa = (unsigned)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(sa));
}
__device__ __forceinline__ unsigned pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // lo in the low half
  return *reinterpret_cast<const unsigned*>(&v);
}
__device__ __forceinline__ void red_add2(float* p, float x, float y) {
  if (x != 0.f || y != 0.f) atomicAdd(reinterpret_cast<float2*>(p), make_float2(x, y));
}

// Batch generator over a warp's range [pos, end) of the concatenated work
// units (per non-empty bucket: kVsBucketCost units, then one per new entry;
// warp-uniform state).
struct VsGen {
  int e, bg;          // current bucket and its (sequence, KV head)
  unsigned pos, end;  // next unit, end of range
  unsigned off0, off1;  // first units of bucket e and e + 1
  unsigned start;     // bucket-local index of the bucket's first new entry
};

// Smallest bucket e' >= e0 whose units hold position x (plan_off
// non-decreasing, plan_off[nent] > x), with its offsets.
// (poff: the exclusive prefix of the round's entries per bucket, in shared
// memory or in the workspace; every bucket's new entries start at 0)
__device__ __forceinline__ void vs_seek(const SparseArgs& a, const unsigned* poff, int nent, int e0, unsigned x,
                                        VsGen& g) {
  const int lane = threadIdx.x & 31;
  for (int base = e0;; base += 32) {
    const int e = base + lane;
    const bool in = e < nent;
    const unsigned o1 = in ? poff[e + 1] : 0xffffffffu;
    const unsigned bal = __ballot_sync(0xffffffffu, o1 > x);
    if (bal) {
      const int f = __ffs(bal) - 1;
      const unsigned o0 = in ? poff[e] : 0u;
      g.e = base + f;
      g.bg = g.e / a.J1;
      g.off0 = __shfl_sync(0xffffffffu, o0, f);
      g.off1 = __shfl_sync(0xffffffffu, o1, f);
      g.start = 0u;
      return;
    }
  }
}

// Buckets up to this count get their gather plan in each value-sum CTA's
// shared memory (no separate plan launch); more use vplan_kernel's.
constexpr int kPlanSmem = 4096;

template <int D, int G>
__global__ void __launch_bounds__(kVsW * 32) vsum_kernel(const SparseArgs a, int nent, int round) {
  pdl_entry();
  using Lt = VsLayout<D, G>;
  constexpr int RB = Lt::RB, MT = Lt::MT, NT = D / 8, CH = RB / 16;
  constexpr int ACC = 2 * D + 8;
  extern __shared__ __align__(16) uint8_t dsm[];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int gq = lane >> 2, tq = lane & 3;
  uint8_t* base = dsm + w * Lt::per_warp;
  uint8_t* s_rows = base + Lt::rows;
  uint8_t* s_sc = base + Lt::sc;
  float* s_vn = reinterpret_cast<float*>(base + Lt::vn);
  uint2* s_ent = reinterpret_cast<uint2*>(base + Lt::ent);
  int* s_desc = reinterpret_cast<int*>(base + Lt::desc);
  uint8_t* s_at = base + Lt::at;
  uint8_t* s_bx = base + Lt::bx;

  // the round's work units per bucket (entries plus kVsBucketCost when
  // non-empty) and their exclusive prefix over the buckets: computed here
  // by every CTA (small plans) or read from vplan_kernel's (large ones)
  const unsigned* poff = a.plan_off;
  if (nent <= kPlanSmem) {
    unsigned* s_plan = reinterpret_cast<unsigned*>(dsm + kVsW * Lt::per_warp);
    __shared__ unsigned s_wsum[kVsW];
    const unsigned* cnt = a.bcnt + (int64_t)round * nent;
    const int nth = kVsW * 32, t = threadIdx.x;
    const int per = (nent + nth - 1) / nth;
    const int i0 = t * per, i1 = min(nent, i0 + per);
    unsigned sum = 0;
    for (int i = i0; i < i1; ++i) {
      const unsigned en = min(cnt[i], (unsigned)a.pcap);
      if (blockIdx.x == 0) a.bcons[i] += en;
      sum += en + (en ? kVsBucketCost : 0u);
    }
    unsigned inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned x = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += x;
    }
    if (lane == 31) s_wsum[w] = inc;
    __syncthreads();
    unsigned wbase = 0, tot = 0;
#pragma unroll
    for (int x = 0; x < kVsW; ++x) {
      if (x < w) wbase += s_wsum[x];
      tot += s_wsum[x];
    }
    unsigned run = wbase + inc - sum;
    for (int i = i0; i < i1; ++i) {
      s_plan[i] = run;
      const unsigned en = min(cnt[i], (unsigned)a.pcap);
      run += en + (en ? kVsBucketCost : 0u);
    }
    if (t == 0) s_plan[nent] = tot;
    __syncthreads();
    poff = s_plan;
  }
  const unsigned E = poff[nent];
  const unsigned nw = gridDim.x * kVsW, gw = blockIdx.x * kVsW + w;
  VsGen gen;
  gen.pos = (unsigned)(((unsigned long long)E * gw) / nw);
  gen.end = (unsigned)(((unsigned long long)E * (gw + 1)) / nw);
  if (gen.pos >= gen.end) return;
  {
    // largest bucket with plan_off <= pos: 32-ary search
    int lo = 0, hi = nent;
    while (hi - lo > 1) {
      const int p = lo + 1 + (int)(((int64_t)(hi - lo - 1) * lane) / 32);
      const unsigned bal = __ballot_sync(0xffffffffu, poff[p] <= gen.pos);
      const int cnt = __popc(bal);
      const int plo = __shfl_sync(0xffffffffu, p, cnt > 0 ? cnt - 1 : 0);
      const int phi = __shfl_sync(0xffffffffu, p, cnt < 32 ? cnt : 31);
      if (cnt == 0) hi = plo;
      else { lo = plo; if (cnt < 32) hi = phi; }
    }
    vs_seek(a, poff, nent, lo, gen.pos, gen);
  }

  // next batch descriptor into slot ds; entries and c32 by cp.async
  auto gen_next = [&](int ds) {
    int* dp = s_desc + ds * 16;
    int cnt = 0, e = -1, bg = 0;
    unsigned eoff = 0;
    if (gen.pos < gen.end) {
      if (gen.pos >= gen.off1) vs_seek(a, poff, nent, gen.e + 1, gen.pos, gen);
      // a bucket's first kVsBucketCost units hold no entries
      const unsigned ent0 = gen.off0 + kVsBucketCost;
      if (gen.pos < ent0) gen.pos = ent0;
      if (gen.pos < gen.end) {
        e = gen.e;
        bg = gen.bg;
        cnt = (int)min(min(gen.off1, gen.end) - gen.pos, (unsigned)kVsB);
        eoff = gen.start + (gen.pos - ent0);
        gen.pos += cnt;
      }
    }
    if (lane == 0) { dp[0] = e; dp[1] = (int)eoff; dp[2] = cnt; dp[3] = bg; }
    if (cnt > 0) {
      const uint2* src = a.buckets + (int64_t)e * a.pcap + eoff;
      if (lane < cnt) cp_async_small<8>(s_ent + ds * kVsB + lane, src + lane, true);
      // query heads of group bg: bh = b * Hq + g * G = bg * G (Hq = G * Hkv)
      if (lane < G) cp_async_small<4>(dp + 4 + lane, a.cmax + ((int64_t)bg * G + lane) * 4 + 3, true);
    }
  };
  // rows, scores and ||v||^2 of batch in descriptor slot ds into stage ss
  auto issue_rows = [&](int ds, int ss) {
    const int* dp = s_desc + ds * 16;
    const int cnt = dp[2];
    if (cnt <= 0) return;
    const int bg = dp[3];
    // lanes 2r and 2r + 1 copy row r (halves of its 16-byte chunks)
    const int r = lane >> 1, half = lane & 1;
    const bool ok = r < cnt;
    const unsigned key = ok ? s_ent[ds * kVsB + r].x : 0u;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(a.V) + ((int64_t)bg * a.n_max + key) * RB +
                         half * (RB / 2);
    uint8_t* dst = s_rows + (ss * kVsB + r) * RB;
#pragma unroll
    for (int i = 0; i < CH / 2; ++i) {
      const int part = half * (CH / 2) + i;
      cp_async16(dst + ((part ^ (r & 7)) << 4), src + i * 16, ok);
    }
    if (half == 0) {
      const float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
      uint8_t* sd = s_sc + (ss * kVsB + r) * Lt::SCB;
      if (G == 8) {
        cp_async16(sd, sp, ok);
        cp_async16(sd + 16, sp + 4, ok);
      } else if (G == 4) {
        cp_async16(sd, sp, ok);
      } else if (G == 2) {
        cp_async_small<8>(sd, sp, ok);
      } else {
        cp_async_small<4>(sd, sp, ok);
      }
    } else {
      cp_async_small<4>(s_vn + ss * kVsB + r, a.vnorm2 + (int64_t)bg * a.n_max + key, ok);
    }
  };

  float C[MT][NT + 1][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int j = 0; j <= NT; ++j) C[mt][j][0] = C[mt][j][1] = C[mt][j][2] = C[mt][j][3] = 0.f;
  int cur = -1, cur_bg = 0;

  auto flush = [&]() {
    const int l = cur - cur_bg * a.J1;
    float* accl = a.acc + ((int64_t)cur_bg * G * a.J1 + l) * ACC;
    const int64_t hstride = (int64_t)a.J1 * ACC;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int row = 16 * mt + gq + 8 * hf;
        if (row >= 4 * G) continue;
        const int type = row / G, h = row - type * G;
        float* ah = accl + h * hstride;
        if (type < 3) {
          const int off = type == 0 ? 0 : D;
#pragma unroll
          for (int j = 0; j < NT; ++j) red_add2(ah + off + 8 * j + 2 * tq, C[mt][j][2 * hf], C[mt][j][2 * hf + 1]);
        }
        // scalar tile: channel 0 = count / weight / sampled, 1 + 2 = ||v||^2 terms
        const float c0 = C[mt][NT][2 * hf], c1 = C[mt][NT][2 * hf + 1];
        if (tq == 0) {
          const int s0 = type == 0 ? 2 * D : (type < 3 ? 2 * D + 2 : 2 * D + 4);
          if (c0 != 0.f) atomicAdd(ah + s0, c0);
          if (type < 3 && c1 != 0.f) atomicAdd(ah + s0 + 1, c1);
        } else if (tq == 1 && type < 3) {
          if (c0 != 0.f) atomicAdd(ah + (type == 0 ? 2 * D + 1 : 2 * D + 3), c0);
        }
      }
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int j = 0; j <= NT; ++j) C[mt][j][0] = C[mt][j][1] = C[mt][j][2] = C[mt][j][3] = 0.f;
  };

  // prologue: descriptors and entries of the first kVsE batches, then rows
  // of the first kVsS
  for (int i = 0; i < kVsE; ++i) gen_next(i);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int i = 0; i < kVsS; ++i) {
    issue_rows(i, i);
    cp_async_commit();
  }
  // coefficient tile of the batch in descriptor slot b_ds / stage b_ss into
  // tile buffer buf: lane k (mod 16) is entry k, lanes 0-15 take heads
  // [0, G/2) and lanes 16-31 heads [G/2, G); branch-free, so it shares a
  // basic block with the previous batch's products
  auto prep = [&](int b_ds, int b_ss, int buf) {
    constexpr int HH = G >= 2 ? G / 2 : 1;
    const int* dq = s_desc + b_ds * 16;
    const int k = lane & 15, hf = lane >> 4;
    const int h0 = G >= 2 ? hf * HH : 0;
    const bool ok = k < dq[2];
    const unsigned m = ok ? s_ent[b_ds * kVsB + k].y : 0u;
    const float* sc = reinterpret_cast<const float*>(s_sc + (b_ss * kVsB + k) * Lt::SCB);
    float cf[HH], wh[HH], wl[HH], ns[HH];
#pragma unroll
    for (int t = 0; t < HH; ++t) {
      const int h = h0 + t;
      const bool add = m & (1u << h), trn = m & (1u << (8 + h)), bef = m & (1u << (16 + h));
      const float x = fsub(sc[h], float_of_ord((unsigned)dq[4 + h]));
      const float wt = trn ? __expf(x) : 0.f;
      cf[t] = add ? 1.f : ((trn && bef) ? -1.f : 0.f);
      wh[t] = __bfloat162float(__float2bfloat16_rn(wt));
      wl[t] = wt - wh[t];
      ns[t] = (add || (trn && !bef)) ? 1.f : 0.f;
    }
    uint8_t* arow = s_at + buf * Lt::atb + k * MT * 32;
    if constexpr (HH >= 2) {
#pragma unroll
      for (int t = 0; t < HH; t += 2) {
        const int e0 = h0 + t;
        *reinterpret_cast<unsigned*>(arow + 2 * (0 * G + e0)) = pack_bf16(cf[t], cf[t + 1]);
        *reinterpret_cast<unsigned*>(arow + 2 * (1 * G + e0)) = pack_bf16(wh[t], wh[t + 1]);
        *reinterpret_cast<unsigned*>(arow + 2 * (2 * G + e0)) = pack_bf16(wl[t], wl[t + 1]);
        *reinterpret_cast<unsigned*>(arow + 2 * (3 * G + e0)) = pack_bf16(ns[t], ns[t + 1]);
      }
    } else {
      *reinterpret_cast<__nv_bfloat16*>(arow + 2 * (0 * G + h0)) = __float2bfloat16_rn(cf[0]);
      *reinterpret_cast<__nv_bfloat16*>(arow + 2 * (1 * G + h0)) = __float2bfloat16_rn(wh[0]);
      *reinterpret_cast<__nv_bfloat16*>(arow + 2 * (2 * G + h0)) = __float2bfloat16_rn(wl[0]);
      *reinterpret_cast<__nv_bfloat16*>(arow + 2 * (3 * G + h0)) = __float2bfloat16_rn(ns[0]);
    }
    const float vn = s_vn[b_ss * kVsB + k];
    const float vh = __bfloat162float(__float2bfloat16_rn(vn));
    *reinterpret_cast<uint4*>(s_bx + buf * kVsB * 16 + k * 16) =
        make_uint4(pack_bf16(1.f, vh), pack_bf16(vn - vh, 0.f), 0u, 0u);
  };
  // rows of A past 4G stay zero in both buffers
  for (int i = lane; i < 2 * Lt::atb / 16; i += 32) reinterpret_cast<uint4*>(s_at)[i] = make_uint4(0u, 0u, 0u, 0u);
  cp_async_wait<kVsS - 1>();
  __syncwarp();
  prep(0, 0, 0);
  for (int i = 0;; ++i) {
    const int ds = i % kVsE, ss = i % kVsS, buf = i & 1;
    const int* dp = s_desc + ds * 16;
    const int e = dp[0], cnt = dp[2];
    if (cnt <= 0) break;
    cp_async_wait<kVsS - 2>();     // rows of batch i + 1 (for its tile)
    __syncwarp();
    if (e != cur) {
      if (cur >= 0) flush();
      cur = e;
      cur_bg = dp[3];
    }
    prep((i + 1) % kVsE, (i + 1) % kVsS, buf ^ 1);
    // A fragments (A^T stored entry-major): matrices (rows m 0-7 | 8-15) x (k 0-7 | 8-15)
    unsigned af[MT][4];
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int k = (mi >> 1) * 8 + rr, mh = mi & 1;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) ldsm_x4_trans(af[mt], s_at + buf * Lt::atb + k * MT * 32 + mt * 32 + mh * 16);
    }
    unsigned bxf[2];
    ldsm_x2_trans(bxf, s_bx + buf * kVsB * 16 + (lane & 15) * 16);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) mma_bf16_16816(C[mt][NT], af[mt], bxf[0], bxf[1]);
    const uint8_t* stg = s_rows + ss * kVsB * RB;
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int ev = (mi & 1) * 8 + rr;
#pragma unroll
      for (int jp = 0; jp < NT / 2; ++jp) {
        const int chunk = 2 * jp + (mi >> 1);
        unsigned bfr[4];
        ldsm_x4_trans(bfr, stg + ev * RB + ((chunk ^ (ev & 7)) << 4));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16_16816(C[mt][2 * jp], af[mt], bfr[0], bfr[1]);
          mma_bf16_16816(C[mt][2 * jp + 1], af[mt], bfr[2], bfr[3]);
        }
      }
    }
    __syncwarp();
    issue_rows((i + kVsS) % kVsE, ss);
    gen_next(ds);
    cp_async_commit();
  }
  cp_async_wait<0>();
  if (cur >= 0) flush();
}

// ------------------------------------------------------------ certificate

template <int D>
__global__ void __launch_bounds__(256) certify_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                      int round) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  constexpr int ACC = 2 * D + 8;
  constexpr int CPL = D / 32;
  constexpr int LB = 32;                   // levels per shared-memory batch
  __shared__ float s_pre[LB][ACC];
  __shared__ float s_vec[LB][4];           // ||c||^2, ||o_hat - c||^2, c.S1, ||o_hat||^2
  __shared__ unsigned s_jr[kMaxJ + 2];     // rows first needed per level (and the 8-bit tier's change)
  __shared__ int s_jd[kMaxJ + 2];
  __shared__ float s_beta[LB], s_dh[LB];
  __shared__ int s_cert[LB];
  __shared__ float s_win[D + 4];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bh = blockIdx.x;
  const int b = bh / a.Hq, hq = bh - b * a.Hq;
  const int G = a.Hq / a.Hkv;
  const int g = hq / G;
  const int bg = b * a.Hkv + g;
  int* st = a.state + (int64_t)bh * 4;
  const int flags = st[3];
  if (flags & kFlagDone) {
    if (round == 0 && (flags & kFlagFallback) && tid == 0) {
      // no pool: exact attention, filled in by the dense pass
      const int64_t n = seq.n[b];
      a.beta[bh] = 0.f; a.level[bh] = 0; a.keys_read[bh] = (int)n;
      if (a.stats) {
        csa_head_stats hs = {0, (int)n, (int)n, 0, 0, 0, 1, (int)n, (int)n, 0};
        a.stats[bh] = hs;
      }
    }
    return;
  }
  const int64_t n = seq.n[b];
  const int J = seq.J[b];
  const int lo = st[0], hi = st[1];
  const float* accb = a.acc + (int64_t)bh * a.J1 * ACC;
  // Thread tid owns columns tid and tid + 256 of the per-level sums: their
  // running totals stay in its registers (r0, r1) across batches and rounds
  // (the previous round's are in pref).  A batch's LB levels are loaded at
  // once, the next batch while this one is evaluated.
  static_assert(ACC <= 512, "two columns per thread");
  const int x0 = tid, x1 = tid + 256;
  const bool h0 = x0 < ACC, h1 = x1 < ACC;
  float v0[LB], v1[LB];
  auto load_batch = [&](int l0, int nl) {
#pragma unroll
    for (int u = 0; u < LB; ++u) {
      v0[u] = (h0 && u < nl) ? accb[(int64_t)(l0 + u) * ACC + x0] : 0.f;
      v1[u] = (h1 && u < nl) ? accb[(int64_t)(l0 + u) * ACC + x1] : 0.f;
    }
  };
  // one round of loads: the first batch, the earlier rounds' sums, the
  // window sums, the rows-needed histogram up to J, the value-norm bound
  int l0 = lo + 1;
  int nl = min(LB, hi - l0 + 1);
  if (l0 <= hi) load_batch(l0, nl);
  float r0 = (h0 && lo >= 0) ? a.pref[(int64_t)bh * ACC + x0] : 0.f;
  float r1 = (h1 && lo >= 0) ? a.pref[(int64_t)bh * ACC + x1] : 0.f;
  for (int i = tid; i < D + 4; i += 256) s_win[i] = a.winstats[(int64_t)bh * (D + 4) + i];
  for (int l = tid; l <= J; l += 256) {
    s_jr[l] = a.jr_hist[(int64_t)bh * (a.J1 + 1) + l];
    s_jd[l] = a.refine8 ? a.jrd[(int64_t)bh * (a.J1 + 1) + l] : 0;
  }
  const float Vp = a.vmaxp[bg];
  __syncthreads();
  const float DR = s_win[D], HR = s_win[D + 1];
  const float de = a.delta / (4.0f * (float)(J + 1));
  const float L = logf(1.0f / de), Lz = logf(2.0f / de);
  int found = -1;
  while (l0 <= hi && found < 0) {
#pragma unroll
    for (int u = 0; u < LB; ++u) {
      if (h0 && u < nl) {
        r0 += v0[u];
        s_pre[u][x0] = r0;
        if (h1) {
          r1 += v1[u];
          s_pre[u][x1] = r1;
        }
      }
    }
    const int l1 = l0 + LB, nl1 = min(LB, hi - l1 + 1);
    if (l1 <= hi) load_batch(l1, nl1);
    __syncthreads();
    // vector parts, one warp per level
    for (int i = w; i < nl; i += 8) {
      const int j = l0 + i;
      const float tau = exp2f(-(float)j / (float)a.r);
      const float* p = s_pre[i];
      const float k = p[2 * D], DB = p[2 * D + 2];
      const float DRB = DR + DB;
      const float Dh = DRB + tau * k;
      float cc = 0.f, oc = 0.f, cs1 = 0.f, oo = 0.f;
#pragma unroll
      for (int x = 0; x < CPL; ++x) {
        const int ch = lane * CPL + x;
        const float nrb = s_win[ch] + p[D + ch];
        const float c = nrb / DRB;
        const float oh = (nrb + tau * p[ch]) / Dh;
        cc += c * c;
        oc += (oh - c) * (oh - c);
        cs1 += c * p[ch];
        oo += oh * oh;
      }
      cc = warp_sum(cc); oc = warp_sum(oc); cs1 = warp_sum(cs1); oo = warp_sum(oo);
      if (lane == 0) { s_vec[i][0] = cc; s_vec[i][1] = oc; s_vec[i][2] = cs1; s_vec[i][3] = oo; }
    }
    __syncthreads();
    // scalar parts, one thread per level
    if (tid < nl) {
      const int i = tid, j = l0 + i;
      const float tau = exp2f(-(float)j / (float)a.r);
      const float* p = s_pre[i];
      const float k = p[2 * D], S2 = p[2 * D + 1], DB = p[2 * D + 2], HB = p[2 * D + 3];
      const float DRB = DR + DB;
      const float Dh = DRB + tau * k;
      const float cc = s_vec[i][0], oc = s_vec[i][1], cs1 = s_vec[i][2], oo = s_vec[i][3];
      float below, above;
      chernoff_gaps(k, Lz, below, above);
      const float dD = tau * fmaxf(below, above);
      const float cn = sqrtf(cc);
      const float Rc = Vp + cn;
      const float Gh = tau * fmaxf(S2 - 2.f * cs1 + k * cc, 0.f);
      const float aa = sqrtf(2.f * tau * Rc * Rc * L);
      const float sq = sqrtf(aa * aa + 4.f * (Gh + (2.f / 3.f) * tau * Rc * Rc * L));
      const float Ghi = 0.25f * (aa + sq) * (aa + sq);
      const float zeta = sqrtf(2.f * tau * Ghi * Lz) + (2.f / 3.f) * tau * Rc * Lz;
      const bool pos = Dh > dD;
      float beta = pos ? (zeta + sqrtf(oc) * dD) / (Dh - dD) : INFINITY;
      bool cert;
      if (a.measure == CSA_MEASURE_CLT) {
        beta = a.zclt * sqrtf(tau * Gh) / Dh;
        const float Mh = sqrtf((HR + HB + tau * S2) / Dh);
        cert = Dh > 0.f && beta <= a.eps * Mh;
      } else if (a.measure == CSA_MEASURE_VALUE) {
        const float Hh = tau * S2;
        const float ap = sqrtf(2.f * tau * Vp * Vp * L);
        const float br = Hh - (2.f / 3.f) * tau * Vp * Vp * L;
        const float t2 = br > 0.f ? 0.5f * (-ap + sqrtf(ap * ap + 4.f * br)) : 0.f;
        const float Dhi = DRB + tau * (k + above);
        const float Mlo = sqrtf((HR + HB + t2 * t2) / Dhi);
        cert = pos && beta <= a.eps * Mlo;
      } else if (a.measure == CSA_MEASURE_OUTPUT) {
        cert = pos && beta * (1.f + a.eps) <= a.eps * sqrtf(oo);
      } else {
        cert = pos && dD <= a.eps * (Dh - dD);
      }
      s_cert[i] = cert;
      s_beta[i] = beta;
      s_dh[i] = Dh;
    }
    __syncthreads();
    for (int i = 0; i < nl; ++i)
      if (s_cert[i]) { found = l0 + i; break; }
    if (found >= 0) {
      const int i = found - l0;
      const float tau = exp2f(-(float)found / (float)a.r);
      const float Dh = s_dh[i];
      for (int c = tid; c < D; c += 256)
        a.o[(int64_t)bh * D + c] = (s_win[c] + s_pre[i][D + c] + tau * s_pre[i][c]) / Dh;
      // rows read up to the stop level: warp 0 sums the bound-level histogram
      unsigned kr = 0, kr8 = 0;
      if (w == 0) {
        for (int l = lane; l <= found; l += 32) {
          kr8 += s_jr[l];
          kr += (unsigned)((int)s_jr[l] + s_jd[l]);
        }
        kr = __reduce_add_sync(0xffffffffu, kr);
        kr8 = __reduce_add_sync(0xffffffffu, kr8);
      }
      if (tid == 0) {
        const int vr = kWindow + (int)s_pre[i][2 * D + 4];
        a.beta[bh] = s_beta[i];
        a.level[bh] = found;
        a.keys_read[bh] = kWindow + (int)kr;
        st[2] = found;
        st[3] = flags | kFlagDone;
        if (a.stats) {
          // 8-bit rows: the candidates outside the head's exact-max set with jbar <= j*
          const int r8 = a.refine8 ? (int)kr8 - (int)a.ninset[bh] : 0;
          csa_head_stats hs = {found, kWindow + (int)kr, vr, (int)a.ncand[bh], 0, J, round + 1,
                               kWindow, kWindow, r8};
          a.stats[bh] = hs;
        }
      }
    }
    __syncthreads();
    l0 = l1;
    nl = nl1;
  }
  if (found < 0 && hi < J) {
    // the head continues: keep its sums through this range for the next round
    if (h0) a.pref[(int64_t)bh * ACC + x0] = r0;
    if (h1) a.pref[(int64_t)bh * ACC + x1] = r1;
  }
  if (found < 0 && tid == 0) {
    if (hi >= J) {
      // no certified level on the grid: exact attention (dense pass)
      a.beta[bh] = 0.f;
      a.level[bh] = J + 1;
      a.keys_read[bh] = (int)n;
      st[2] = J + 1;
      st[3] = flags | kFlagDone | kFlagFallback;
      atomicAdd(a.nfall, 1u);
      if (a.stats) {
        csa_head_stats hs = {J + 1, (int)n, (int)n, (int)a.ncand[bh], 0, J, round + 1, kWindow, kWindow, 0};
        a.stats[bh] = hs;
      }
    } else {
      int nh = (round == 0) ? hi + 2 * a.r : J;
      st[0] = hi;
      st[1] = nh > J ? J : nh;
      if (round < 2) rq_push(a, round + 1, bg);
    }
  }
}

// --------------------------------------------------- near-threshold count

template <int G>
__global__ void __launch_bounds__(256) near_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq_arg) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow || !a.stats) return;
  const int64_t P = n - kWindow;
  const int64_t key = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const int bh0 = b * a.Hq + g * G;
  const int J = seq.J[b];
  const float neg_r = -(float)a.r;
  bool needK = false, needV = false;
  if (key < P) {
    const float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
    const float* ub = a.ubar + ((int64_t)bg * a.n_max + key) * G;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float t = a.per_head ? a.t32[((int64_t)bg * a.pcap + key) * G + h] : a.t32[(int64_t)bg * a.pcap + key];
      const int js = a.state[(int64_t)(bh0 + h) * 4 + 2];
      if (js > J) { needK = needV = true; continue; }   // exact fallback
      if (js < 0) continue;
      const float u = ub[h];
      int jb = bound_level(u, cmax_get(a, bh0 + h, 2), t, neg_r, J);
      // the 8-bit tier: a refined candidate is needed from its refined level
      if (a.refine8 && jb <= J && u < cmax_get(a, bh0 + h, 0) &&
          (a.jkey[(int64_t)bg * a.pcap + key] & 0x200u))
        jb = a.jref[((int64_t)bg * a.pcap + key) * G + h];
      if (u >= cmax_get(a, bh0 + h, 0) || jb <= js) needK = true;
      const float s = sp[h];
      if (!(s > -INFINITY)) continue;
      int jl, hl;
      exact_levels(s, cmax_get(a, bh0 + h, 3), t, neg_r, J, jl, hl);
      if (jl <= js) needV = true;
      // keys within 1e-5 nats of the light or heavy threshold at the stop
      const float dl = fsub(s, cmax_get(a, bh0 + h, 3));
      const float thr = -((float)js / (float)a.r) * 0.69314718f;
      const float x = dl + t * 0.69314718f;
      if (fabsf(x - thr) < 1e-5f || fabsf(dl - thr) < 1e-5f)
        atomicAdd(&a.stats[bh0 + h].n_near_threshold, 1);
    }
  }
  const int ck = __popc(__ballot_sync(0xffffffffu, needK));
  const int cv = __popc(__ballot_sync(0xffffffffu, needV));
  if (lane == 0 && (ck || cv)) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (ck) atomicAdd(&a.stats[bh0 + h].group_keys_read, ck);
      if (cv) atomicAdd(&a.stats[bh0 + h].group_values_read, cv);
    }
  }
}

// --------------------------------------------------------------- launches

#define CSA_DG_SWITCH(FN, ...)                                                                   \
  switch (d * 100 + G * 10 + (bf16 ? 1 : 0)) {                                                   \
    case 12811: FN<128, 1, __nv_bfloat16> __VA_ARGS__; break;                                    \
    case 12821: FN<128, 2, __nv_bfloat16> __VA_ARGS__; break;                                    \
    case 12841: FN<128, 4, __nv_bfloat16> __VA_ARGS__; break;                                    \
    case 12881: FN<128, 8, __nv_bfloat16> __VA_ARGS__; break;                                    \
    case 12810: FN<128, 1, float> __VA_ARGS__; break;                                            \
    case 12820: FN<128, 2, float> __VA_ARGS__; break;                                            \
    case 12840: FN<128, 4, float> __VA_ARGS__; break;                                            \
    case 12880: FN<128, 8, float> __VA_ARGS__; break;                                            \
    case 6411: FN<64, 1, __nv_bfloat16> __VA_ARGS__; break;                                      \
    case 6421: FN<64, 2, __nv_bfloat16> __VA_ARGS__; break;                                      \
    case 6441: FN<64, 4, __nv_bfloat16> __VA_ARGS__; break;                                      \
    case 6481: FN<64, 8, __nv_bfloat16> __VA_ARGS__; break;                                      \
    case 6410: FN<64, 1, float> __VA_ARGS__; break;                                              \
    case 6420: FN<64, 2, float> __VA_ARGS__; break;                                              \
    case 6440: FN<64, 4, float> __VA_ARGS__; break;                                              \
    case 6480: FN<64, 8, float> __VA_ARGS__; break;                                              \
    default: return cudaErrorInvalidValue;                                                       \
  }

#define CSA_DG_LAUNCH(FN, ...)                                                                   \
  switch (d * 100 + G * 10 + (bf16 ? 1 : 0)) {                                                   \
    case 12811: launch_pdl(FN<128, 1, __nv_bfloat16>, __VA_ARGS__); break;                                    \
    case 12821: launch_pdl(FN<128, 2, __nv_bfloat16>, __VA_ARGS__); break;                                    \
    case 12841: launch_pdl(FN<128, 4, __nv_bfloat16>, __VA_ARGS__); break;                                    \
    case 12881: launch_pdl(FN<128, 8, __nv_bfloat16>, __VA_ARGS__); break;                                    \
    case 12810: launch_pdl(FN<128, 1, float>, __VA_ARGS__); break;                                            \
    case 12820: launch_pdl(FN<128, 2, float>, __VA_ARGS__); break;                                            \
    case 12840: launch_pdl(FN<128, 4, float>, __VA_ARGS__); break;                                            \
    case 12880: launch_pdl(FN<128, 8, float>, __VA_ARGS__); break;                                            \
    case 6411: launch_pdl(FN<64, 1, __nv_bfloat16>, __VA_ARGS__); break;                                      \
    case 6421: launch_pdl(FN<64, 2, __nv_bfloat16>, __VA_ARGS__); break;                                      \
    case 6441: launch_pdl(FN<64, 4, __nv_bfloat16>, __VA_ARGS__); break;                                      \
    case 6481: launch_pdl(FN<64, 8, __nv_bfloat16>, __VA_ARGS__); break;                                      \
    case 6410: launch_pdl(FN<64, 1, float>, __VA_ARGS__); break;                                              \
    case 6420: launch_pdl(FN<64, 2, float>, __VA_ARGS__); break;                                              \
    case 6440: launch_pdl(FN<64, 4, float>, __VA_ARGS__); break;                                              \
    case 6480: launch_pdl(FN<64, 8, float>, __VA_ARGS__); break;                                              \
    default: return cudaErrorInvalidValue;                                                       \
  }

#define CSA_G_SWITCH(FN, ...)                                                                    \
  switch (G) {                                                                                   \
    case 1: launch_pdl(FN<1>, __VA_ARGS__); break;                                               \
    case 2: launch_pdl(FN<2>, __VA_ARGS__); break;                                               \
    case 4: launch_pdl(FN<4>, __VA_ARGS__); break;                                               \
    case 8: launch_pdl(FN<8>, __VA_ARGS__); break;                                               \
    default: return cudaErrorInvalidValue;                                                       \
  }

// CTAs per (b, g) group: `target` CTAs shared out over the groups (at
// least 1, at most `cap`)
static int per_group(const SparseArgs& a, int64_t target, int64_t cap) {
  int64_t per = (target + a.B * a.Hkv - 1) / (a.B * a.Hkv);
  if (per > cap) per = cap;
  return per < 1 ? 1 : (int)per;
}

template <int D, int G, typename E, int MODE>
void launch_rows_t(int64_t items, int nsm, cudaStream_t st, const SparseArgs& a, const SeqArgs& seq, int round) {
  constexpr int smem = rows_smem<D, G, E>();
  cudaFuncSetAttribute(rows_kernel<D, G, E, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  // kRowsCps (16) CTAs of 4 warps per SM over all groups, several waves:
  // many short shares balance the uneven density of wanted entries (and
  // keep more rows in flight) better than one long share per resident warp
  // (rescoring of the unsplit 128K x 4 step: 199 us with 4 CTAs of 8 warps
  // per SM; 179, 168 and 164 us with 8, 12 and 16 CTAs of 4 warps)
  const int per = per_group(a, (MODE == 0 ? kRows0Cps : kRowsCps) * (int64_t)nsm, (items + 8 * kRingW - 1) / (8 * kRingW));
  launch_pdl(rows_kernel<D, G, E, MODE>, dim3((unsigned)per, (unsigned)(a.B * a.Hkv)), dim3(kRingW * 32), smem, st,
             a, seq, round);
}
template <int D, int G, typename E>
void launch_rows0(int64_t items, int nsm, cudaStream_t st, const SparseArgs& a, const SeqArgs& seq) {
  launch_rows_t<D, G, E, 0>(items, nsm, st, a, seq, 0);
}
template <int D, int G, typename E>
void launch_rows1(int64_t items, int nsm, cudaStream_t st, const SparseArgs& a, const SeqArgs& seq, int round) {
  launch_rows_t<D, G, E, 1>(items, nsm, st, a, seq, round);
}
template <int G>
void launch_cand_t(int64_t pmax, int nsm, cudaStream_t st, const SparseArgs& a, const SeqArgs& seq) {
  const int smem = cand_smem(G, a.J1);
  cudaFuncSetAttribute(cand_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  const int64_t span = (int64_t)kTile * kTilesPerCta;
  dim3 grid((unsigned)((pmax + span - 1) / span), (unsigned)(a.B * a.Hkv));
  launch_pdl(cand_kernel<G>, grid, dim3(256), smem, st, a, seq, (int)span);
}
template <int G>
void launch_cset_t(int64_t nmax, int nsm, cudaStream_t st, const SparseArgs& a, const SeqArgs& seq) {
  const int64_t span = 256 * kCsetTiles;
  dim3 grid((unsigned)((nmax + span - 1) / span), (unsigned)(a.B * a.Hkv));
  launch_pdl(cset_kernel<G>, grid, dim3(256), 0, st, a, seq, (int)span);
}
template <int D, int G, typename E>
void launch_vgather_t(int nsm, cudaStream_t st, const SparseArgs& a, const SeqArgs& seq, int nent, int round,
                      PhaseMark mark) {
  if constexpr (sizeof(E) == 2) {
    const bool small = nent <= kPlanSmem;
    const int smem = VsLayout<D, G>::smem + (small ? (nent + 1) * 4 : 0);
    cudaFuncSetAttribute(vsum_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    // resident CTAs per SM: a property of the device and the shared memory
    // size, looked up once per (device, size) (the query costs host time on
    // every step otherwise)
    static int occ_dev[64] = {0}, occ_smem[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int per_sm = occ_smem[dev] == smem ? occ_dev[dev] : 0;
    if (per_sm < 1) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, vsum_kernel<D, G>, kVsW * 32, smem) !=
              cudaSuccess ||
          per_sm < 1)
        per_sm = 1;
      occ_dev[dev] = per_sm;
      occ_smem[dev] = smem;
    }
    if (!small) {
      launch_pdl(vplan_kernel<true>, dim3(1), dim3(1024), 0, st, a, nent, round);
      add_launches(1);
    }
    if (mark) mark(7, st);
    launch_pdl(vsum_kernel<D, G>, dim3((unsigned)(nsm * per_sm)), dim3(kVsW * 32), smem, st, a, nent, round);
  } else {
    constexpr int smem = vgather_smem<D, G, E>();
    cudaFuncSetAttribute(vgather_kernel<D, G, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    launch_pdl(vplan_kernel<false>, dim3(1), dim3(1024), 0, st, a, nent, round);
    add_launches(1);
    if (mark) mark(7, st);
    launch_pdl(vgather_kernel<D, G, E>, dim3((unsigned)(nsm * 2)), dim3(256), smem, st, a, seq, nent);
  }
}

cudaError_t launch_cstar(const SparseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, int64_t nmax_live,
                         int nsm, cudaStream_t st) {
  switch (G) {
    case 1: launch_cset_t<1>(nmax_live, nsm, st, a, seq); break;
    case 2: launch_cset_t<2>(nmax_live, nsm, st, a, seq); break;
    case 4: launch_cset_t<4>(nmax_live, nsm, st, a, seq); break;
    case 8: launch_cset_t<8>(nmax_live, nsm, st, a, seq); break;
    default: return cudaErrorInvalidValue;
  }
  CSA_DG_SWITCH(launch_rows0, (nmax_live, nsm, st, a, seq))
  return cudaGetLastError();
}
cudaError_t launch_candidates(const SparseArgs& a, const SeqArgs& seq, int G, int64_t pmax_live, int nsm,
                              cudaStream_t st) {
  switch (G) {
    case 1: launch_cand_t<1>(pmax_live, nsm, st, a, seq); break;
    case 2: launch_cand_t<2>(pmax_live, nsm, st, a, seq); break;
    case 4: launch_cand_t<4>(pmax_live, nsm, st, a, seq); break;
    case 8: launch_cand_t<8>(pmax_live, nsm, st, a, seq); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}
cudaError_t launch_predict(const SparseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, cudaStream_t st) {
  dim3 grid((unsigned)(a.B * a.Hkv));
  CSA_DG_LAUNCH(predict_kernel, grid, dim3(256), 0, st, a, seq)
  return cudaGetLastError();
}
template <int D, int G>
static cudaError_t launch_refine_t(const SparseArgs& a, const SeqArgs& seq, int round, int nsm, cudaStream_t st) {
  const int smem = RfLayout<D, G>::hist + G * (a.J1 + 1) * 4;
  const cudaError_t e = cudaFuncSetAttribute(refine8_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per = per_group(a, 4 * (int64_t)nsm, (a.nblk_max + kRfW - 1) / kRfW);
  launch_pdl(refine8_kernel<D, G>, dim3((unsigned)per, (unsigned)(a.B * a.Hkv)), dim3(kRfW * 32), smem, st, a, seq,
             round);
  return cudaGetLastError();
}

cudaError_t launch_round(const SparseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, int64_t pmax_live,
                         int round, int nsm, cudaStream_t st, PhaseMark mark) {
  if (a.refine8) {
    // the 8-bit refinement of the round's candidates (bf16 caches only)
    cudaError_t e = cudaErrorInvalidValue;
    switch (d * 10 + G) {
      case 1281: e = launch_refine_t<128, 1>(a, seq, round, nsm, st); break;
      case 1282: e = launch_refine_t<128, 2>(a, seq, round, nsm, st); break;
      case 1284: e = launch_refine_t<128, 4>(a, seq, round, nsm, st); break;
      case 1288: e = launch_refine_t<128, 8>(a, seq, round, nsm, st); break;
      case 641: e = launch_refine_t<64, 1>(a, seq, round, nsm, st); break;
      case 642: e = launch_refine_t<64, 2>(a, seq, round, nsm, st); break;
      case 644: e = launch_refine_t<64, 4>(a, seq, round, nsm, st); break;
      case 648: e = launch_refine_t<64, 8>(a, seq, round, nsm, st); break;
      default: break;
    }
    if (e != cudaSuccess) return e;
    add_launches(1);
    if (mark) mark(12, st);
  }
  // kLevCps 256-thread CTAs per SM pull work items (isz keys of a group
  // listed for this round) from the round's queue
  const int isz = round == 0 ? kLevItem : kLevItemLate;
  const unsigned tpg = (unsigned)((pmax_live + isz - 1) / isz);
  int64_t nct = kLevCps * (int64_t)nsm;
  const int64_t items = (int64_t)tpg * a.B * a.Hkv;
  if (nct > items) nct = items;
  if (nct < 1) nct = 1;
  dim3 grid((unsigned)nct);
  CSA_DG_SWITCH(launch_rows1, (pmax_live, nsm, st, a, seq, round))
  if (mark) mark(4, st);
  switch (G * 2 + (a.per_head ? 1 : 0)) {
    case 2: launch_pdl(levels_kernel<1, false>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    case 3: launch_pdl(levels_kernel<1, true>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    case 4: launch_pdl(levels_kernel<2, false>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    case 5: launch_pdl(levels_kernel<2, true>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    case 8: launch_pdl(levels_kernel<4, false>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    case 9: launch_pdl(levels_kernel<4, true>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    case 16: launch_pdl(levels_kernel<8, false>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    case 17: launch_pdl(levels_kernel<8, true>, grid, dim3(256), 0, st, a, seq, round, tpg, isz); break;
    default: return cudaErrorInvalidValue;
  }
  if (mark) mark(6, st);
  const int nent = a.B * a.Hkv * a.J1;
  CSA_DG_SWITCH(launch_vgather_t, (nsm, st, a, seq, nent, round, mark))
  if (mark) mark(8, st);
  dim3 cg((unsigned)(a.B * a.Hq));
  if (d == 128) launch_pdl(certify_kernel<128>, cg, dim3(256), 0, st, a, seq, round);
  else launch_pdl(certify_kernel<64>, cg, dim3(256), 0, st, a, seq, round);
  if (mark) mark(9, st);
  return cudaGetLastError();
}
cudaError_t launch_near(const SparseArgs& a, const SeqArgs& seq, int G, int64_t pmax_live, cudaStream_t st) {
  dim3 grid((unsigned)((pmax_live + 255) / 256), (unsigned)(a.B * a.Hkv));
  CSA_G_SWITCH(near_kernel, grid, dim3(256), 0, st, a, seq)
  return cudaGetLastError();
}

}  // namespace csa
