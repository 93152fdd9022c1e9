// Dense decode attention (picx.dev "Problem Setup": o = sum_i w_i v_i / sum_i
// w_i, w_i = exp(s_i - c*)), float32 throughout.  It is the same-build
// comparator of the sparse step, and the exact fallback of the sparse step
// for heads with no certified level (and for sequences with no pool).
//
// Split-K over the keys: a CTA takes 1024 keys of one (sequence, KV head)
// for all G query heads; each warp scores eight K rows at a time (one row
// load serves the G heads; lane-local products then an eight-row shuffle
// reduction), keeps an online-softmax state per head and accumulates the
// eight V rows.  The K and V rows come through a per-warp ring of
// shared-memory stages filled with cp.async, kDenseStages batches ahead.
// A second kernel merges the splits.
#include "csa_args.cuh"

namespace csa {

constexpr int kDenseChunk = 1024;

// ring stages per warp: 8 K rows and 8 V rows each (bf16: three stages, so
// two CTAs fit an SM; 2, 3 and 4 stages gave 625, 612 and 682 us for the
// 128K x 4 comparator)
template <typename E>
__host__ __device__ constexpr int dense_stages() { return sizeof(E) == 2 ? 3 : 2; }
template <int D, typename E>
__host__ __device__ constexpr int dense_smem() { return 8 * dense_stages<E>() * 2 * 8 * D * (int)sizeof(E); }

// stage the 8 consecutive rows [k0, k0 + 8) of K and V (rows >= end are
// zero-filled) with 16-byte cp.async copies
template <int D, typename E>
__device__ __forceinline__ void dense_stage(uint8_t* dk, uint8_t* dv, const E* Kb, const E* Vb, int64_t k0,
                                            int64_t end) {
  constexpr int RB = D * (int)sizeof(E);
  constexpr int CH = RB / 16;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = lane; c < 8 * CH; c += 32) {
    const int r = c / CH, part = c - r * CH;
    const bool ok = k0 + r < end;
    const int64_t off = ok ? (k0 + r) * RB + part * 16 : 0;
    cp_async16(dk + r * RB + part * 16, reinterpret_cast<const uint8_t*>(Kb) + off, ok);
    cp_async16(dv + r * RB + part * 16, reinterpret_cast<const uint8_t*>(Vb) + off, ok);
  }
}

template <int D, typename E>
__device__ __forceinline__ void dload_row(const E* row, float* v) {
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

__device__ __forceinline__ bool group_wanted(const DenseArgs& a, int b, int g, int G) {
  if (!a.state) return true;
  for (int h = 0; h < G; ++h)
    if (a.state[((int64_t)b * a.Hq + g * G + h) * 4 + 3] & 1) return true;
  return false;
}

template <int D, int G, typename E>
__global__ void __launch_bounds__(256) dense_split_kernel(const DenseArgs a, const __grid_constant__ SeqArgs seq_arg,
                                                          int nsplit_live) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  constexpr int CPL = D / 32;
  constexpr int S = dense_stages<E>();
  constexpr int RB = D * (int)sizeof(E);
  __shared__ float s_m[8][G], s_l[8][G];
  __shared__ float s_acc[8][G][D];
  extern __shared__ __align__(16) uint8_t dsm[];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  uint8_t* ringk = dsm + w * S * 2 * 8 * RB;          // [S][8 rows] of K, then of V
  uint8_t* ringv = ringk + S * 8 * RB;
  if (a.nfall && *a.nfall == 0u) return;
  const int nitems = nsplit_live * a.B * a.Hkv;
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
  const int split = item % nsplit_live;
  const int bg = item / nsplit_live, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  const int64_t start = (int64_t)split * kDenseChunk;
  if (start >= n) continue;
  if (!group_wanted(a, b, g, G)) continue;
  const int64_t end = min(n, start + kDenseChunk);
  float qv[G][CPL];
  const E* qp = reinterpret_cast<const E*>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * G) * D;
#pragma unroll
  for (int h = 0; h < G; ++h) dload_row<D, E>(qp + (int64_t)h * D, qv[h]);
  float m[G], l[G], acc[G][CPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY; l[h] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[h][c] = 0.f;
  }
  const E* Kb = reinterpret_cast<const E*>(a.K) + (int64_t)bg * a.n_max * D;
  const E* Vb = reinterpret_cast<const E*>(a.V) + (int64_t)bg * a.n_max * D;
  // this warp's batches: rows [start + 8w + 64i, + 8) for i < nb
  const int64_t first = start + w * 8;
  const int nb = first < end ? (int)((end - first + 63) / 64) : 0;
#pragma unroll
  for (int i = 0; i < S; ++i) {
    if (i < nb) dense_stage<D, E>(ringk + i * 8 * RB, ringv + i * 8 * RB, Kb, Vb, first + 64 * i, end);
    cp_async_commit();
  }
  for (int i = 0; i < nb; ++i) {
    const int64_t k0 = first + 64 * i;
    const int slot = i % S;
    cp_async_wait<S - 1>();
    __syncwarp();
    float kv[8][CPL], vv[8][CPL];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      dload_row<D, E>(reinterpret_cast<const E*>(ringk + (slot * 8 + r) * RB), kv[r]);
      dload_row<D, E>(reinterpret_cast<const E*>(ringv + (slot * 8 + r) * RB), vv[r]);
    }
    __syncwarp();
    // refill the slot with the batch S ahead
    if (i + S < nb)
      dense_stage<D, E>(ringk + slot * 8 * RB, ringv + slot * 8 * RB, Kb, Vb, first + 64 * (i + S), end);
    cp_async_commit();
    const bool valid = k0 + (lane & 7) < end;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float part[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        float p[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) p[c] = kv[r][c] * qv[h][c];
        part[r] = local_tree<CPL>(p);
      }
      float s = reduce8_rows(part) * a.rs;
      if (!valid) s = -INFINITY;
      float m8 = s;
      m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 1));
      m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 2));
      m8 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 4));
      const float mn = fmaxf(m[h], m8);
      const float sc = expf(m[h] - mn);
      const float p = expf(s - mn);
      float ps = p;
      ps += __shfl_xor_sync(0xffffffffu, ps, 1);
      ps += __shfl_xor_sync(0xffffffffu, ps, 2);
      ps += __shfl_xor_sync(0xffffffffu, ps, 4);
      l[h] = l[h] * sc + ps;
      m[h] = mn;
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[h][c] *= sc;
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float pr = __shfl_sync(0xffffffffu, p, r);
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[h][c] += pr * vv[r][c];
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) { s_m[w][h] = m[h]; s_l[w][h] = l[h]; }
#pragma unroll
    for (int c = 0; c < CPL; ++c) s_acc[w][h][lane * CPL + c] = acc[h][c];
  }
  __syncthreads();
  for (int i = tid; i < G * (D + 2); i += 256) {
    const int h = i / (D + 2), c = i - h * (D + 2);
    float M = -INFINITY;
#pragma unroll
    for (int x = 0; x < 8; ++x) M = fmaxf(M, s_m[x][h]);
    float v = 0.f;
    if (c == 0) v = M;
    else {
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const float e = s_m[x][h] > -INFINITY ? expf(s_m[x][h] - M) : 0.f;
        v += e * (c == 1 ? s_l[x][h] : s_acc[x][h][c - 2]);
      }
    }
    a.part[((int64_t)split * a.B * a.Hq + (int64_t)b * a.Hq + g * G + h) * (D + 2) + c] = v;
  }
  __syncthreads();
  }
}

template <int D>
__global__ void __launch_bounds__(128) dense_combine_kernel(const DenseArgs a, const __grid_constant__ SeqArgs seq_arg) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  const int bh = blockIdx.x;
  const int b = bh / a.Hq;
  if (a.nfall && *a.nfall == 0u) return;
  if (a.state && !(a.state[(int64_t)bh * 4 + 3] & 1)) return;
  const int64_t n = seq.n[b];
  const int ns = (int)((n + kDenseChunk - 1) / kDenseChunk);
  const int64_t stride = (int64_t)a.B * a.Hq * (D + 2);
  const float* p = a.part + (int64_t)bh * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, p[s * stride]);
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float num = 0.f, den = 0.f;
    for (int s = 0; s < ns; ++s) {
      const float e = expf(p[s * stride] - M);
      den += e * p[s * stride + 1];
      num += e * p[s * stride + 2 + c];
    }
    a.o[(int64_t)bh * D + c] = num / den;
  }
}

// ------------------------------------------- tensor-core dense (bf16 caches)
//
// The same split-K decomposition (one work item = 1024 keys of one
// (sequence, KV head) for its G query heads, partials merged by
// dense_combine_kernel), with the tiles moved by the tensor memory
// accelerator and the two products on tensor cores:
//  * a producer warp streams 64-key tiles of K and V into a ring of
//    kDtStages shared-memory stages with 2-D bulk tensor copies (boxes of
//    64 keys x 64 channels, 128-byte swizzle), each stage completing on an
//    mbarrier with its byte count; consumers release a stage on a second
//    mbarrier;
//  * four consumer warps take 16 keys of each tile: S = Q K^T with
//    mma.sync m16n8k16 (rows = the group's query heads, padded to 16;
//    K fragments by ldmatrix from the swizzled stage), an online softmax per
//    head, and O^T += V^T P^T (rows = channels, columns = heads; V
//    fragments by ldmatrix.trans, P split into bf16 hi + lo parts so the
//    weights keep ~16 bits);
//  * at the end of an item the four warps' states merge in shared memory
//    into one partial (m, l, acc[D]) per head.
// Keys past the item's end are masked (score -inf) and their V rows zeroed
// in shared memory before use (the box reads whatever lies there).
constexpr int kDtKeys = 64;      // keys per tile
constexpr int kDtStages = 4;     // ring stages
constexpr int kDtWarps = 4;      // consumer warps (16 keys of each tile)

template <int D>
struct DtLayout {
  static constexpr int BOX = kDtKeys * 128;             // one 64-key x 64-channel box
  static constexpr int TILE = kDtKeys * D * 2;          // a K or V tile (D / 64 boxes)
  static constexpr int STAGE = 2 * TILE;                // K, then V
  static constexpr int bars = kDtStages * STAGE;        // full[S], empty[S]
  static constexpr int fm = bars + 2 * kDtStages * 8;   // m [W][8], l [W][8]
  static constexpr int fo = fm + kDtWarps * 8 * 4 * 2;  // o [W][8][D]
  static constexpr int end = fo + kDtWarps * 8 * D * 4;
  static constexpr int smem = end + 1024;               // + alignment of the base
};

// byte offset of 16-byte chunk c of row r in a swizzled tile
__device__ __forceinline__ unsigned dt_off(int r, int c) {
  return (unsigned)((c >> 3) * (kDtKeys * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void dt_ldsm_x4(unsigned (&r)[4], unsigned addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void dt_ldsm_x4_t(unsigned (&r)[4], unsigned addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void dt_mma(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                       unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned dt_pack(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const unsigned*>(&v);
}

// the work items of this CTA, in order; false for items with nothing to do
__device__ __forceinline__ bool dt_item(const DenseArgs& a, const SeqArgs& seq, int G, int nsplit, int item,
                                        int& bg, int& split, int64_t& start, int64_t& end) {
  split = item % nsplit;
  bg = item / nsplit;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  start = (int64_t)split * kDenseChunk;
  if (start >= n) return false;
  if (!group_wanted(a, b, g, G)) return false;
  end = min(n, start + kDenseChunk);
  return true;
}

template <int D, int G>
__global__ void __launch_bounds__((kDtWarps + 1) * 32) dense_tc_kernel(const DenseArgs a,
                                                                       const __grid_constant__ SeqArgs seq_arg,
                                                                       const __grid_constant__ CUtensorMap tmK,
                                                                       const __grid_constant__ CUtensorMap tmV,
                                                                       int nsplit_live) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  using Lt = DtLayout<D>;
  constexpr int KS = D / 16;     // k-steps of S = Q K^T (channels)
  constexpr int MT = D / 16;     // m-tiles of O^T (channels)
  constexpr int NB = D / 64;     // boxes per row
  extern __shared__ __align__(16) uint8_t dsm_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  const unsigned sbase = smem_u32(sm);
  const unsigned bar_full = sbase + Lt::bars, bar_empty = bar_full + kDtStages * 8;
  float* s_m = reinterpret_cast<float*>(sm + Lt::fm);
  float* s_l = s_m + kDtWarps * 8;
  float* s_o = reinterpret_cast<float*>(sm + Lt::fo);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (a.nfall && *a.nfall == 0u) return;
  if (tid == 0) {
    for (int s = 0; s < kDtStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kDtWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int nitems = nsplit_live * a.B * a.Hkv;
  bool dead = false;   // a bounded wait gave up: finish the control flow, skip waits

  if (w == kDtWarps) {
    // ------------------------------------------------------- producer
    if (lane == 0) {
      int t = 0;
      for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        int bg, split;
        int64_t start, end;
        if (!dt_item(a, seq, G, nsplit_live, item, bg, split, start, end)) continue;
        const int ntile = (int)((end - start + kDtKeys - 1) / kDtKeys);
        for (int k = 0; k < ntile; ++k, ++t) {
          const int s = t % kDtStages;
          if (t >= kDtStages && !dead && !mbar_wait(bar_empty + 8 * s, ((t / kDtStages) - 1) & 1)) dead = true;
          if (dead) continue;
          const unsigned st = sbase + s * Lt::STAGE;
          mbar_expect_tx(bar_full + 8 * s, Lt::STAGE);
          const int row = (int)((int64_t)bg * a.n_max + start + (int64_t)k * kDtKeys);
#pragma unroll
          for (int bx = 0; bx < NB; ++bx) {
            tma_load_2d(st + bx * Lt::BOX, &tmK, 64 * bx, row, bar_full + 8 * s);
            tma_load_2d(st + Lt::TILE + bx * Lt::BOX, &tmV, 64 * bx, row, bar_full + 8 * s);
          }
        }
      }
      // the CTA stays until the copies it started have landed
      for (int i = max(0, t - kDtStages); i < t; ++i)
        if (!mbar_wait(bar_full + 8 * (i % kDtStages), (i / kDtStages) & 1)) dead = true;
      if (dead && a.status) atomicOr(a.status, 4u);
    }
    return;
  }

  // --------------------------------------------------------- consumers
  const int tq = lane & 3;
  const int hr = lane >> 2;                 // row of S / head this lane's softmax state belongs to
  const int mi = lane >> 3, li = lane & 7;  // ldmatrix: matrix and row this lane addresses
  const int lrow = 16 * w + (mi >> 1) * 8 + li;
  int t = 0;
  int cur_bg = -1;
  unsigned qa[KS][2];
  for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
    int bg, split;
    int64_t start, end;
    if (!dt_item(a, seq, G, nsplit_live, item, bg, split, start, end)) continue;
    const int b = bg / a.Hkv, g = bg - b * a.Hkv;
    if (bg != cur_bg) {
      // A fragments of Q (rows = heads; rows >= G and 8..15 are zero)
      const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                ((int64_t)b * a.Hq + (int64_t)g * G + (hr < G ? hr : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = hr < G ? *reinterpret_cast<const unsigned*>(qp + 16 * ks + 2 * tq) : 0u;
        qa[ks][1] = hr < G ? *reinterpret_cast<const unsigned*>(qp + 16 * ks + 2 * tq + 8) : 0u;
      }
      cur_bg = bg;
    }
    float m = -INFINITY, l = 0.f;
    float oacc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
    const int ntile = (int)((end - start + kDtKeys - 1) / kDtKeys);
    for (int k = 0; k < ntile; ++k, ++t) {
      const int s = t % kDtStages;
      if (!dead && !mbar_wait(bar_full + 8 * s, (t / kDtStages) & 1)) dead = true;
      const unsigned kt = sbase + s * Lt::STAGE, vt = kt + Lt::TILE;
      const int64_t kbase = start + (int64_t)k * kDtKeys + 16 * w;
      const int nvalid = (int)max((int64_t)0, min((int64_t)16, end - kbase));
      if (nvalid < 16) {
        // rows past the item's end: zero their V rows (their scores are masked)
        for (int c = lane; c < 16 * (D / 8); c += 32) {
          const int r = c / (D / 8), cc = c - r * (D / 8);
          if (r >= nvalid) {
            const unsigned adr = vt + dt_off(16 * w + r, cc);
            asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};\n" ::"r"(adr), "r"(0u) : "memory");
          }
        }
        fence_proxy_async();
        __syncwarp();
      }
      // S = Q K^T for this warp's 16 keys: two n-tiles of 8 keys
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        unsigned bf[4];
        dt_ldsm_x4(bf, kt + dt_off(lrow, 2 * ks + (mi & 1)));
        dt_mma(sacc[0], qa[ks][0], 0u, qa[ks][1], 0u, bf[0], bf[1]);
        dt_mma(sacc[1], qa[ks][0], 0u, qa[ks][1], 0u, bf[2], bf[3]);
      }
      // online softmax of head hr over the 16 keys (lanes 4hr..4hr+3 hold
      // keys 2tq, 2tq+1 of each n-tile)
      float sv[2][2];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = 8 * j + 2 * tq + e;
          sv[j][e] = kk < nvalid ? sacc[j][e] * a.rs : -INFINITY;
          mx = fmaxf(mx, sv[j][e]);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m, mx);
      float sc = 1.f, p[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      if (mn > -INFINITY) {
        const float L2E = 1.4426950408889634f;
        sc = exp2f((m - mn) * L2E);
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) p[j][e] = exp2f((sv[j][e] - mn) * L2E);
      }
      float ps = (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
      ps += __shfl_xor_sync(0xffffffffu, ps, 1);
      ps += __shfl_xor_sync(0xffffffffu, ps, 2);
      l = l * sc + ps;
      m = mn;
      // O^T columns of this lane are heads 2tq, 2tq+1: their scale factors
      const float sc0 = __shfl_sync(0xffffffffu, sc, 8 * tq);
      const float sc1 = __shfl_sync(0xffffffffu, sc, 8 * tq + 4);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        oacc[mt][0] *= sc0; oacc[mt][1] *= sc1;
        oacc[mt][2] *= sc0; oacc[mt][3] *= sc1;
      }
      // P^T (keys x heads) as the B operand: hi and lo bf16 parts
      const unsigned bh0 = dt_pack(p[0][0], p[0][1]), bh1 = dt_pack(p[1][0], p[1][1]);
      const float2 h0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bh0));
      const float2 h1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bh1));
      const unsigned bl0 = dt_pack(p[0][0] - h0.x, p[0][1] - h0.y);
      const unsigned bl1 = dt_pack(p[1][0] - h1.x, p[1][1] - h1.y);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        unsigned af[4];
        dt_ldsm_x4_t(af, vt + dt_off(lrow, 2 * mt + (mi & 1)));
        dt_mma(oacc[mt], af[0], af[1], af[2], af[3], bh0, bh1);
        dt_mma(oacc[mt], af[0], af[1], af[2], af[3], bl0, bl1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    // merge the four warps' states into the item's partial per head
    if (tq == 0 && hr < G) { s_m[w * 8 + hr] = m; s_l[w * 8 + hr] = l; }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * tq + e;
          if (h < G) s_o[(w * 8 + h) * D + 16 * mt + hr + 8 * hf] = oacc[mt][2 * hf + e];
        }
    bar_sync(1, kDtWarps * 32);
    for (int i = tid; i < G * (D + 2); i += kDtWarps * 32) {
      const int h = i / (D + 2), c = i - h * (D + 2);
      float M = -INFINITY;
#pragma unroll
      for (int x = 0; x < kDtWarps; ++x) M = fmaxf(M, s_m[x * 8 + h]);
      float v = M;
      if (c > 0) {
        v = 0.f;
#pragma unroll
        for (int x = 0; x < kDtWarps; ++x) {
          const float mx_ = s_m[x * 8 + h];
          const float e = mx_ > -INFINITY ? expf(mx_ - M) : 0.f;
          v += e * (c == 1 ? s_l[x * 8 + h] : s_o[(x * 8 + h) * D + c - 2]);
        }
      }
      a.part[((int64_t)split * a.B * a.Hq + (int64_t)b * a.Hq + g * G + h) * (D + 2) + c] = v;
    }
    bar_sync(1, kDtWarps * 32);
  }
  if (dead && a.status && lane == 0) atomicOr(a.status, 4u);
}

#define CSA_DENSE_SWITCH(FN, ...)                                                                \
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

int dense_nsplit(int64_t n_max) { return (int)((n_max + kDenseChunk - 1) / kDenseChunk); }

// opt in to the ring's dynamic shared memory.  Done on every launch: the
// attribute belongs to the function in the current context, so a flag kept
// per process would be wrong on a second device or after a device reset,
// and the call is cheap.
template <int D, typename E>
cudaError_t set_dense_smem(int G) {
  const int smem = dense_smem<D, E>();
  switch (G) {
    case 1: return cudaFuncSetAttribute(dense_split_kernel<D, 1, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 2: return cudaFuncSetAttribute(dense_split_kernel<D, 2, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 4: return cudaFuncSetAttribute(dense_split_kernel<D, 4, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 8: return cudaFuncSetAttribute(dense_split_kernel<D, 8, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    default: return cudaErrorInvalidValue;
  }
}

template <int D, int G>
cudaError_t launch_dense_tc_t(const DenseArgs& a, const SeqArgs& seq, int nsplit_live, int nct,
                              const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  constexpr int smem = DtLayout<D>::smem;
  cudaError_t e = cudaFuncSetAttribute(dense_tc_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  launch_pdl(dense_tc_kernel<D, G>, dim3((unsigned)nct), dim3((kDtWarps + 1) * 32), smem, st, a, seq, tk, tv,
             nsplit_live);
  return cudaGetLastError();
}

// bf16 caches: the tensor-core kernel when the tensor maps can be made
// (16-byte aligned caches and fewer than 2^31 rows), one CTA per SM over
// the work items; returns cudaErrorNotSupported otherwise
static cudaError_t launch_dense_tc(const DenseArgs& a, const SeqArgs& seq, int d, int G, int nsplit_live,
                                   cudaStream_t st) {
  const uint64_t rows = (uint64_t)a.B * a.Hkv * (uint64_t)a.n_max;
  if (rows >= (1ull << 31)) return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  if (!make_tmap_2d_bf16(&tk, a.K, (uint64_t)d, rows, (uint64_t)d * 2, 64, kDtKeys) ||
      !make_tmap_2d_bf16(&tv, a.V, (uint64_t)d, rows, (uint64_t)d * 2, 64, kDtKeys))
    return cudaErrorNotSupported;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm < 1)
    nsm = 148;
  const int items = nsplit_live * a.B * a.Hkv;
  const int nct = items < nsm ? items : nsm;
  switch (d * 10 + G) {
    case 1281: return launch_dense_tc_t<128, 1>(a, seq, nsplit_live, nct, tk, tv, st);
    case 1282: return launch_dense_tc_t<128, 2>(a, seq, nsplit_live, nct, tk, tv, st);
    case 1284: return launch_dense_tc_t<128, 4>(a, seq, nsplit_live, nct, tk, tv, st);
    case 1288: return launch_dense_tc_t<128, 8>(a, seq, nsplit_live, nct, tk, tv, st);
    case 641: return launch_dense_tc_t<64, 1>(a, seq, nsplit_live, nct, tk, tv, st);
    case 642: return launch_dense_tc_t<64, 2>(a, seq, nsplit_live, nct, tk, tv, st);
    case 644: return launch_dense_tc_t<64, 4>(a, seq, nsplit_live, nct, tk, tv, st);
    case 648: return launch_dense_tc_t<64, 8>(a, seq, nsplit_live, nct, tk, tv, st);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_dense(const DenseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, int64_t nmax_live,
                         cudaStream_t st) {
  const int nsplit_live = (int)((nmax_live + kDenseChunk - 1) / kDenseChunk);
  if (bf16) {
    const cudaError_t e = launch_dense_tc(a, seq, d, G, nsplit_live, st);
    if (e == cudaSuccess) {
      if (d == 128) launch_pdl(dense_combine_kernel<128>, dim3(a.B * a.Hq), dim3(128), 0, st, a, seq);
      else launch_pdl(dense_combine_kernel<64>, dim3(a.B * a.Hq), dim3(128), 0, st, a, seq);
      return cudaGetLastError();
    }
    if (e != cudaErrorNotSupported) return e;
  }
  int items = nsplit_live * a.B * a.Hkv;
  // comparator: one CTA per item; fallback (masked): a small persistent grid
  const int cap = a.state ? 1024 : items;
  dim3 grid((unsigned)(items < cap ? items : cap));
  const cudaError_t ea = d == 128 ? (bf16 ? set_dense_smem<128, __nv_bfloat16>(G) : set_dense_smem<128, float>(G))
                                  : (bf16 ? set_dense_smem<64, __nv_bfloat16>(G) : set_dense_smem<64, float>(G));
  if (ea != cudaSuccess) return ea;
  const int smem = d == 128 ? (bf16 ? dense_smem<128, __nv_bfloat16>() : dense_smem<128, float>())
                            : (bf16 ? dense_smem<64, __nv_bfloat16>() : dense_smem<64, float>());
  CSA_DENSE_SWITCH(dense_split_kernel, grid, dim3(256), smem, st, a, seq, nsplit_live)
  if (d == 128) launch_pdl(dense_combine_kernel<128>, dim3(a.B * a.Hq), dim3(128), 0, st, a, seq);
  else launch_pdl(dense_combine_kernel<64>, dim3(a.B * a.Hq), dim3(128), 0, st, a, seq);
  return cudaGetLastError();
}

}  // namespace csa
