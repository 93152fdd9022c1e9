// The sparse part of the decode step, after the 4-bit scan.
//
// picx.dev summary, "Algorithm Components" 1-4 and Theorem 4; readsearch.ai
// "Abstract".  Kernels, in launch order, for every (sequence b, KV head g):
//   cstar_kernel    exact maximum: float32 rescoring of the window and of the
//                   pool keys with ubar >= c*_lo; c32 = max score, and the
//                   certified lower bound cb = max fl(s32 - fl(mag * 2^-13))
//   rescore_kernel  perturbations t_i, bound levels jbar_i, candidates
//                   (jbar <= J); exact float32 scores of candidate K rows (one
//                   row load serves the G heads); per-level counts and heavy
//                   weights that need no values
//   predict_kernel  window sums (D_R, N_R, H_R) and, from the value-free
//                   per-level counts, a predicted stop level per head that
//                   sizes the first gather round
//   levels_kernel   (per round) exact inclusion / heavy levels; each key that
//                   changes a head's sums at a level of the round is appended
//                   once to the (b, g, level) bucket
//   vplan_kernel    (per round) chunk list over the new bucket entries
//   vgather_kernel  (per round) V rows of the bucketed keys; per-level
//                   Horvitz-Thompson sums (light count, sum v, sum ||v||^2;
//                   heavy sum w, sum w v, sum w ||v||^2) accumulated per head
//   certify_kernel  (per round) prefix over levels, Chernoff interval,
//                   Bernstein bound on G, Pinelis bound zeta, beta, value
//                   scale lower bound; first certified level -> outputs
//   near_kernel     optional diagnostics: near-threshold keys at the stop
#include "csa_args.cuh"

namespace csa {

constexpr int kFlagFallback = 1;
constexpr int kFlagDone = 2;
constexpr int kChunk = 1024;   // bucket entries per gather work item

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

// Scores of eight rows (float32, adjacent-pair tree, times rs) for G heads.
// rows[r] null -> zero row.  On return lane l holds in s[h] the score of row
// (l & 7) and, when MAG, in m[h] the tree sum of |products| times rs.
template <int D, int G, typename E, bool MAG>
__device__ __forceinline__ void score8(const E* const rows[8], const float (&qv)[G][D / 32], float rs,
                                       float (&s)[G], float (&m)[G]) {
  constexpr int CPL = D / 32;
  float kv[8][CPL];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if (rows[r]) load_row<D, E>(rows[r], kv[r]);
    else {
#pragma unroll
      for (int c = 0; c < CPL; ++c) kv[r][c] = 0.f;
    }
  }
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
      pm[r] = local_tree<CPL>(pa);
    }
    s[h] = fmul(reduce8_rows(part), rs);
    if (MAG) m[h] = fmul(reduce8_rows(pm), rs);
  }
}

// Chernoff interval for a Poisson-binomial count k (two-sided, budget
// delta_e / 2 per side): mu = k e^y with e^y - 1 - y = Lz / k.  Returns
// k - mu_lo and mu_hi - k (both >= 0), bracket ends taken outward.
__device__ __forceinline__ float phi_y(float y) {
  if (fabsf(y) < 0.05f) return y * y * (0.5f + y * (1.0f / 6.0f + y * (1.0f / 24.0f + y * (1.0f / 120.0f))));
  return expm1f(y) - y;
}
__device__ void chernoff_gaps(float k, float Lz, float& below, float& above) {
  if (!(k > 0.f)) { below = 0.f; above = Lz; return; }
  float c0 = Lz / k;
  // upper root, y > 0
  float lo = 0.f, hi = fmaxf(1.0f, logf(3.0f * c0 + 3.0f));
  for (int it = 0; it < 8 && phi_y(hi) < c0; ++it) hi *= 2.0f;
  for (int it = 0; it < 48; ++it) {
    float mid = 0.5f * (lo + hi);
    if (phi_y(mid) <= c0) lo = mid; else hi = mid;
  }
  above = k * expm1f(hi);
  // lower root, y < 0
  float a = -(c0 + 1.0f), b2 = 0.f;
  for (int it = 0; it < 48; ++it) {
    float mid = 0.5f * (a + b2);
    if (phi_y(mid) > c0) a = mid; else b2 = mid;
  }
  below = -k * expm1f(a);
}

// ----------------------------------------------------------------- c* step

template <int D, int G, typename E>
__global__ void __launch_bounds__(256) cstar_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq) {
  constexpr int CPL = D / 32;
  __shared__ int s_list[kTile];
  __shared__ unsigned s_qm[kTile];
  __shared__ int s_cnt;
  __shared__ float s_cb[8][G], s_c32[8][G];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  const int64_t key0 = (int64_t)blockIdx.x * kTile;
  if (key0 >= n) return;
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  const int bh0 = b * a.Hq + g * G;
  {
    const int64_t key = key0 + tid;
    unsigned qm = 0;
    if (key < n) {
      if (key >= P) qm = (1u << G) - 1u;
      else {
        const float* ub = a.ubar + ((int64_t)bg * a.n_max + key) * G;
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (ub[h] >= cmax_get(a, bh0 + h, 0)) qm |= 1u << h;
      }
    }
    if (qm) {
      int p = atomicAdd(&s_cnt, 1);
      s_list[p] = (int)(key - key0);
      s_qm[p] = qm;
    }
  }
  __syncthreads();
  const int cnt = s_cnt;
  float qv[G][CPL];
  {
    const E* qp = reinterpret_cast<const E*>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * G) * D;
#pragma unroll
    for (int h = 0; h < G; ++h) load_row<D, E>(qp + (int64_t)h * D, qv[h]);
  }
  float cbm[G], c3m[G];
#pragma unroll
  for (int h = 0; h < G; ++h) { cbm[h] = -INFINITY; c3m[h] = -INFINITY; }
  const E* Kb = reinterpret_cast<const E*>(a.K) + (int64_t)bg * a.n_max * D;
  for (int base = w * 8; base < cnt; base += 64) {
    const E* rows[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      rows[r] = (base + r < cnt) ? Kb + (key0 + s_list[base + r]) * D : nullptr;
    float s[G], m[G];
    score8<D, G, E, true>(rows, qv, a.rs, s, m);
    const int r = lane & 7;
    if (lane < 8 && base + r < cnt) {
      const int64_t key = key0 + s_list[base + r];
      const unsigned qm = s_qm[base + r];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (qm & (1u << h)) {
          cbm[h] = fmaxf(cbm[h], fsub(s[h], fmul(m[h], 1.220703125e-04f)));   // 2^-13
          c3m[h] = fmaxf(c3m[h], s[h]);
        }
      }
      if (key >= P) {
        float* wp = a.win + ((int64_t)bg * kWindow + (key - P)) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) wp[h] = s[h];
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float x = warp_max(cbm[h]), y = warp_max(c3m[h]);
    if (lane == 0) { s_cb[w][h] = x; s_c32[w][h] = y; }
  }
  __syncthreads();
  if (tid < G) {
    float x = -INFINITY, y = -INFINITY;
    for (int i = 0; i < 8; ++i) { x = fmaxf(x, s_cb[i][tid]); y = fmaxf(y, s_c32[i][tid]); }
    if (x > -INFINITY) atomic_max_f(a.cmax + (int64_t)(bh0 + tid) * 4 + 2, x);
    if (y > -INFINITY) atomic_max_f(a.cmax + (int64_t)(bh0 + tid) * 4 + 3, y);
  }
}

// ------------------------------------------------- candidates + rescoring

template <int D, int G, typename E>
__global__ void __launch_bounds__(256) rescore_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq) {
  constexpr int CPL = D / 32;
  __shared__ int s_list[kTile];
  __shared__ unsigned s_cm[kTile];
  __shared__ float s_t[kTile];
  __shared__ int s_cnt;
  __shared__ unsigned s_jr[G][kMaxJ + 2];
  __shared__ unsigned s_nc[G];
  __shared__ float s_pre[G][kMaxJ + 1][3];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  const int64_t key0 = (int64_t)blockIdx.x * kTile;
  if (key0 >= P) return;
  const int J = seq.J[b];
  const float neg_r = -(float)a.r;
  for (int i = tid; i < G * (kMaxJ + 2); i += 256) (&s_jr[0][0])[i] = 0u;
  for (int i = tid; i < G * (J + 1) * 3; i += 256) {
    int h = i / ((J + 1) * 3), rem = i - h * (J + 1) * 3;
    s_pre[h][rem / 3][rem % 3] = 0.f;
  }
  if (tid < G) s_nc[tid] = 0u;
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  const int bh0 = b * a.Hq + g * G;
  const unsigned long long gk = group_key(seq.seed[b], g);
  {
    const int64_t key = key0 + tid;
    unsigned cm = 0;
    if (key < P) {
      const float t = perturb_t(gk, key);
      const float* ub = a.ubar + ((int64_t)bg * a.n_max + key) * G;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float u = ub[h];
        const int jb = bound_level(u, cmax_get(a, bh0 + h, 2), t, neg_r, J);
        const bool cand = jb <= J;
        const bool inc = u >= cmax_get(a, bh0 + h, 0);
        const int jr = inc ? 0 : (cand ? jb : J + 1);
        atomicAdd(&s_jr[h][jr], 1u);
        if (cand) { cm |= 1u << h; atomicAdd(&s_nc[h], 1u); }
      }
      if (cm) {
        int p = atomicAdd(&s_cnt, 1);
        s_list[p] = tid;
        s_cm[p] = cm;
        s_t[p] = t;
      } else {
        float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) sp[h] = -INFINITY;
      }
    }
  }
  __syncthreads();
  const int cnt = s_cnt;
  float qv[G][CPL];
  {
    const E* qp = reinterpret_cast<const E*>(a.q) + ((int64_t)b * a.Hq + (int64_t)g * G) * D;
#pragma unroll
    for (int h = 0; h < G; ++h) load_row<D, E>(qp + (int64_t)h * D, qv[h]);
  }
  float c32[G];
#pragma unroll
  for (int h = 0; h < G; ++h) c32[h] = cmax_get(a, bh0 + h, 3);
  const E* Kb = reinterpret_cast<const E*>(a.K) + (int64_t)bg * a.n_max * D;
  for (int base = w * 8; base < cnt; base += 64) {
    const E* rows[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
      rows[r] = (base + r < cnt) ? Kb + (key0 + s_list[base + r]) * D : nullptr;
    float s[G], m[G];
    score8<D, G, E, false>(rows, qv, a.rs, s, m);
    const int r = lane & 7;
    if (lane < 8 && base + r < cnt) {
      const int64_t key = key0 + s_list[base + r];
      const unsigned cm = s_cm[base + r];
      const float t = s_t[base + r];
      float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const bool c = cm & (1u << h);
        sp[h] = c ? s[h] : -INFINITY;
        if (c) {
          int jl, hl;
          exact_levels(s[h], c32[h], t, neg_r, J, jl, hl);
          if (jl <= J) atomicAdd(&s_pre[h][jl][2], 1.0f);
          if (jl < hl) {
            atomicAdd(&s_pre[h][jl][0], 1.0f);
            if (hl <= J) atomicAdd(&s_pre[h][hl][0], -1.0f);
          }
          if (hl <= J) atomicAdd(&s_pre[h][hl][1], expf(fsub(s[h], c32[h])));
        }
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < G * (J + 2); i += 256) {
    int h = i / (J + 2), l = i - h * (J + 2);
    unsigned v = s_jr[h][l];
    if (v) atomicAdd(a.jr_hist + (int64_t)(bh0 + h) * (a.J1 + 1) + l, v);
  }
  for (int i = tid; i < G * (J + 1) * 3; i += 256) {
    int h = i / ((J + 1) * 3), rem = i - h * (J + 1) * 3;
    float v = s_pre[h][rem / 3][rem % 3];
    if (v != 0.f) atomicAdd(a.pre_hist + ((int64_t)(bh0 + h) * a.J1 + rem / 3) * 4 + rem % 3, v);
  }
  if (tid < G && s_nc[tid]) atomicAdd(a.ncand + bh0 + tid, s_nc[tid]);
}

// -------------------------------------------- window sums + stop predictor

template <int D, int G, typename E>
__global__ void __launch_bounds__(256) predict_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq) {
  constexpr int CPL = D / 32;
  __shared__ float s_nr[G][D];
  __shared__ float s_dr[G], s_hr[G];
  __shared__ float s_vm[8];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int bg = blockIdx.x, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  const int bh0 = b * a.Hq + g * G;
  if (n <= kWindow) {
    // no pool: dense attention for every head of the group
    if (tid < G) {
      int* st = a.state + (int64_t)(bh0 + tid) * 4;
      st[0] = 0; st[1] = 0; st[2] = 0; st[3] = kFlagFallback | kFlagDone;
    }
    return;
  }
  const int64_t P = n - kWindow;
  const int J = seq.J[b];
  for (int i = tid; i < G * D; i += 256) (&s_nr[0][0])[i] = 0.f;
  if (tid < G) { s_dr[tid] = 0.f; s_hr[tid] = 0.f; }
  __syncthreads();
  float c32[G];
#pragma unroll
  for (int h = 0; h < G; ++h) c32[h] = cmax_get(a, bh0 + h, 3);
  const E* Vb = reinterpret_cast<const E*>(a.V) + ((int64_t)bg * a.n_max + P) * D;
  float nr[G][CPL], dr[G], hr[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    dr[h] = 0.f; hr[h] = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) nr[h][c] = 0.f;
  }
  for (int row = w; row < kWindow; row += 8) {
    float v[CPL];
    load_row<D, E>(Vb + (int64_t)row * D, v);
    float sq = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) sq += v[c] * v[c];
    const float* ws = a.win + ((int64_t)bg * kWindow + row) * G;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float wt = expf(fsub(ws[h], c32[h]));
      dr[h] += wt;
      hr[h] += wt * sq;
#pragma unroll
      for (int c = 0; c < CPL; ++c) nr[h][c] += wt * v[c];
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) atomicAdd(&s_nr[h][lane * CPL + c], nr[h][c]);
    float hs = warp_sum(hr[h]);
    if (lane == 0) { atomicAdd(&s_dr[h], dr[h]); atomicAdd(&s_hr[h], hs); }
  }
  // largest value-norm bound over the pool blocks
  {
    const int64_t nbp = (P + kBlock - 1) / kBlock;
    float m = 0.f;
    for (int64_t i = tid; i < nbp; i += 256) m = fmaxf(m, a.vmax[(int64_t)bg * a.nblk_max + i]);
    m = warp_max(m);
    if (lane == 0) s_vm[w] = m;
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
    float runk = 0.f, rundb = 0.f;
    int pred = J;
    for (int l0 = 0; l0 <= J; l0 += 32) {
      const int j = l0 + lane;
      float dk = 0.f, ddb = 0.f;
      if (j <= J) {
        const float* ph = a.pre_hist + ((int64_t)bh * a.J1 + j) * 4;
        dk = ph[0]; ddb = ph[1];
      }
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
      unsigned bal = __ballot_sync(0xffffffffu, pass);
      if (bal) { pred = l0 + __ffs(bal) - 1; break; }
    }
    if (lane == 0) {
      int hi = pred + (a.r + 1) / 2;
      if (hi > J) hi = J;
      int* st = a.state + (int64_t)bh * 4;
      st[0] = -1; st[1] = hi; st[2] = -1; st[3] = 0;
    }
  }
}

// --------------------------------------------------------- level buckets

template <int G>
__global__ void __launch_bounds__(256) levels_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq) {
  __shared__ unsigned s_cnt[kMaxJ + 1];
  __shared__ unsigned s_base[kMaxJ + 1];
  __shared__ int s_any;
  const int tid = threadIdx.x;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow) return;
  const int64_t P = n - kWindow;
  const int64_t key0 = (int64_t)blockIdx.x * kTile;
  if (key0 >= P) return;
  const int J = seq.J[b];
  const int bh0 = b * a.Hq + g * G;
  int lo[G], hi[G];
  bool any = false;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int* st = a.state + (int64_t)(bh0 + h) * 4;
    lo[h] = st[0];
    hi[h] = (st[3] & kFlagDone) ? st[0] : st[1];
    any |= hi[h] > lo[h];
  }
  if (!any) return;
  for (int i = tid; i <= J; i += 256) s_cnt[i] = 0u;
  __syncthreads();
  const float neg_r = -(float)a.r;
  const int64_t key = key0 + tid;
  int ev[2 * G], pos[2 * G];
  int nev = 0;
  if (key < P) {
    const float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
    float s[G];
    bool some = false;
#pragma unroll
    for (int h = 0; h < G; ++h) { s[h] = sp[h]; some |= s[h] > -INFINITY; }
    if (some) {
      const float t = perturb_t(group_key(seq.seed[b], g), key);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (!(s[h] > -INFINITY)) continue;
        int jl, hl;
        exact_levels(s[h], cmax_get(a, bh0 + h, 3), t, neg_r, J, jl, hl);
        int c1 = (jl < hl && jl > lo[h] && jl <= hi[h]) ? jl : -1;
        int c2 = (hl <= J && hl > lo[h] && hl <= hi[h]) ? hl : -1;
        int cs[2] = {c1, c2};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (cs[e] < 0) continue;
          bool dup = false;
          for (int x = 0; x < nev; ++x) dup |= ev[x] == cs[e];
          if (!dup) ev[nev++] = cs[e];
        }
      }
    }
  }
  for (int x = 0; x < nev; ++x) pos[x] = (int)atomicAdd(&s_cnt[ev[x]], 1u);
  __syncthreads();
  for (int i = tid; i <= J; i += 256)
    if (s_cnt[i]) s_base[i] = atomicAdd(a.bcnt + (int64_t)bg * a.J1 + i, s_cnt[i]);
  __syncthreads();
  for (int x = 0; x < nev; ++x) {
    const int l = ev[x];
    const unsigned p = s_base[l] + (unsigned)pos[x];
    if (p < (unsigned)a.pcap)
      a.buckets[((int64_t)bg * a.J1 + l) * a.pcap + p] = (unsigned)key;
    else
      atomicOr(a.status, 2u);
  }
}

// One CTA: chunk list over the bucket entries appended since the last plan.
__global__ void __launch_bounds__(1024) vplan_kernel(const SparseArgs a, int nent) {
  __shared__ unsigned s_part[1024];
  const int tid = threadIdx.x;
  const int per = (nent + 1023) / 1024;
  const int i0 = tid * per, i1 = min(nent, i0 + per);
  unsigned sum = 0;
  for (int i = i0; i < i1; ++i) {
    unsigned st = a.bcons[i], en = a.bcnt[i];
    if (en > (unsigned)a.pcap) en = (unsigned)a.pcap;
    a.plan_start[i] = st;
    a.plan_end[i] = en;
    a.bcons[i] = en;
    sum += (en - st + kChunk - 1) / kChunk;
  }
  s_part[tid] = sum;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    unsigned x = tid >= o ? s_part[tid - o] : 0u;
    __syncthreads();
    s_part[tid] += x;
    __syncthreads();
  }
  unsigned run = s_part[tid] - sum;
  for (int i = i0; i < i1; ++i) {
    a.plan_off[i] = run;
    run += (a.plan_end[i] - a.plan_start[i] + kChunk - 1) / kChunk;
  }
  if (tid == 1023) a.plan_off[nent] = s_part[1023];
}

// ------------------------------------------------------------- V gather

template <int D, int G, typename E>
__global__ void __launch_bounds__(256) vgather_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq,
                                                      int nent) {
  constexpr int CPL = D / 32;
  constexpr int ACC = 2 * D + 8;
  __shared__ float s_acc[G][ACC];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const unsigned total = a.plan_off[nent];
  const float neg_r = -(float)a.r;
  for (unsigned c = blockIdx.x; c < total; c += gridDim.x) {
    // find the (b, g, level) entry of chunk c
    int lo_e = 0, hi_e = nent - 1;
    while (lo_e < hi_e) {
      int mid = (lo_e + hi_e + 1) >> 1;
      if (a.plan_off[mid] <= c) lo_e = mid; else hi_e = mid - 1;
    }
    const int e = lo_e;
    const int bg = e / a.J1, l = e - bg * a.J1;
    const int b = bg / a.Hkv, g = bg - b * a.Hkv;
    const int bh0 = b * a.Hq + g * G;
    const int J = seq.J[b];
    const unsigned ev0 = a.plan_start[e] + (c - a.plan_off[e]) * kChunk;
    const unsigned ev1 = min(a.plan_end[e], ev0 + kChunk);
    unsigned hm = 0;
    float c32[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int* st = a.state + (int64_t)(bh0 + h) * 4;
      if (!(st[3] & kFlagDone) && l > st[0] && l <= st[1]) hm |= 1u << h;
      c32[h] = cmax_get(a, bh0 + h, 3);
    }
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
    const unsigned* bk = a.buckets + (int64_t)e * a.pcap;
    const E* Vb = reinterpret_cast<const E*>(a.V) + (int64_t)bg * a.n_max * D;
    const float* sb = a.s32 + (int64_t)bg * a.pcap * G;
    const unsigned long long gk = group_key(seq.seed[b], g);
    for (unsigned base = ev0 + w * 32; base < ev1 && hm; base += 256) {
      // lane-parallel per-event bookkeeping
      const unsigned my = base + lane;
      unsigned key = 0, msk = 0;
      float wl[G];
#pragma unroll
      for (int h = 0; h < G; ++h) wl[h] = 0.f;
      if (my < ev1) {
        key = bk[my];
        const float t = perturb_t(gk, key);
        const float* sp = sb + (int64_t)key * G;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (!(hm & (1u << h))) continue;
          const float s = sp[h];
          if (!(s > -INFINITY)) continue;
          int jl, hl;
          exact_levels(s, c32[h], t, neg_r, J, jl, hl);
          const bool add = (jl == l) && (jl < hl);
          const bool trn = (hl == l);
          const bool bef = jl < hl;
          if (add) { msk |= 1u << h; kc[h] += 1.f; }
          if (trn) {
            msk |= 1u << (8 + h);
            if (bef) { msk |= 1u << (16 + h); kc[h] -= 1.f; }
            wl[h] = expf(fsub(s, c32[h]));
            db[h] += wl[h];
          }
          if (jl == l) ns[h] += 1.f;
        }
      }
      const int cntw = (int)min(32u, ev1 - base);
      for (int j0 = 0; j0 < cntw; j0 += 4) {
        float v[4][CPL];
        unsigned mk[4];
        float wv[4][G];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u;
          const unsigned kk = __shfl_sync(0xffffffffu, key, j & 31);
          mk[u] = __shfl_sync(0xffffffffu, msk, j & 31);
#pragma unroll
          for (int h = 0; h < G; ++h) wv[u][h] = __shfl_sync(0xffffffffu, wl[h], j & 31);
          if (j < cntw && mk[u]) load_row<D, E>(Vb + (int64_t)kk * D, v[u]);
          else {
            mk[u] = 0;
#pragma unroll
            for (int x = 0; x < CPL; ++x) v[u][x] = 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (!mk[u]) continue;
          float sq = 0.f;
#pragma unroll
          for (int x = 0; x < CPL; ++x) sq += v[u][x] * v[u][x];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if (mk[u] & (1u << h)) {
#pragma unroll
              for (int x = 0; x < CPL; ++x) S1[h][x] += v[u][x];
              s2[h] += sq;
            }
            if (mk[u] & (1u << (8 + h))) {
              if (mk[u] & (1u << (16 + h))) {
#pragma unroll
                for (int x = 0; x < CPL; ++x) S1[h][x] -= v[u][x];
                s2[h] -= sq;
              }
              const float ww = wv[u][h];
#pragma unroll
              for (int x = 0; x < CPL; ++x) NB[h][x] += ww * v[u][x];
              hb[h] += ww * sq;
            }
          }
        }
      }
    }
    // fold the warp's sums into the CTA, then into the per-level sums
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (!(hm & (1u << h))) continue;
#pragma unroll
      for (int x = 0; x < CPL; ++x) {
        atomicAdd(&s_acc[h][lane * CPL + x], S1[h][x]);
        atomicAdd(&s_acc[h][D + lane * CPL + x], NB[h][x]);
      }
      const float k_ = warp_sum(kc[h]), s2_ = warp_sum(s2[h]), db_ = warp_sum(db[h]);
      const float hb_ = warp_sum(hb[h]), ns_ = warp_sum(ns[h]);
      if (lane == 0) {
        atomicAdd(&s_acc[h][2 * D + 0], k_);
        atomicAdd(&s_acc[h][2 * D + 1], s2_);
        atomicAdd(&s_acc[h][2 * D + 2], db_);
        atomicAdd(&s_acc[h][2 * D + 3], hb_);
        atomicAdd(&s_acc[h][2 * D + 4], ns_);
      }
    }
    __syncthreads();
    for (int i = tid; i < G * ACC; i += 256) {
      const int h = i / ACC, x = i - h * ACC;
      if (!(hm & (1u << h)) || x >= 2 * D + 5) continue;
      const float v = s_acc[h][x];
      if (v != 0.f) atomicAdd(a.acc + ((int64_t)(bh0 + h) * a.J1 + l) * ACC + x, v);
    }
  }
}

// ------------------------------------------------------------ certificate

template <int D>
__global__ void __launch_bounds__(256) certify_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq,
                                                      int round) {
  constexpr int ACC = 2 * D + 8;
  constexpr int CPL = D / 32;
  constexpr int LB = 32;                   // levels per shared-memory batch
  __shared__ float s_pre[LB][ACC];
  __shared__ float s_run[ACC];
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
        csa_head_stats hs = {0, (int)n, (int)n, 0, 0, 0, 1, 0};
        a.stats[bh] = hs;
      }
    }
    return;
  }
  const int64_t n = seq.n[b];
  const int J = seq.J[b];
  const int lo = st[0], hi = st[1];
  for (int i = tid; i < D + 4; i += 256) s_win[i] = a.winstats[(int64_t)bh * (D + 4) + i];
  for (int x = tid; x < ACC; x += 256) s_run[x] = 0.f;
  __syncthreads();
  const float DR = s_win[D], HR = s_win[D + 1];
  const float Vp = a.vmaxp[bg];
  const float de = a.delta / (4.0f * (float)(J + 1));
  const float L = logf(1.0f / de), Lz = logf(2.0f / de);
  const float* accb = a.acc + (int64_t)bh * a.J1 * ACC;
  int found = -1;
  // prefix up to lo (levels already known not to certify)
  for (int x = tid; x < ACC; x += 256) {
    float run = 0.f;
    for (int l = 0; l <= lo; ++l) run += accb[(int64_t)l * ACC + x];
    s_run[x] = run;
  }
  __syncthreads();
  for (int l0 = lo + 1; l0 <= hi && found < 0; l0 += LB) {
    const int nl = min(LB, hi - l0 + 1);
    for (int x = tid; x < ACC; x += 256) {
      float run = s_run[x];
      for (int i = 0; i < nl; ++i) {
        run += accb[(int64_t)(l0 + i) * ACC + x];
        s_pre[i][x] = run;
      }
      s_run[x] = run;
    }
    __syncthreads();
    for (int i = w; i < nl; i += 8) {
      const int j = l0 + i;
      const float tau = exp2f(-(float)j / (float)a.r);
      const float* p = s_pre[i];
      const float k = p[2 * D], S2 = p[2 * D + 1], DB = p[2 * D + 2], HB = p[2 * D + 3];
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
      if (lane == 0) {
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
        const float beta = pos ? (zeta + sqrtf(oc) * dD) / (Dh - dD) : INFINITY;
        bool cert;
        if (a.measure == CSA_MEASURE_VALUE) {
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
      if (tid == 0) {
        const unsigned* jr = a.jr_hist + (int64_t)bh * (a.J1 + 1);
        unsigned kr = 0;
        for (int l = 0; l <= found; ++l) kr += jr[l];
        const int vr = kWindow + (int)s_pre[i][2 * D + 4];
        a.beta[bh] = s_beta[i];
        a.level[bh] = found;
        a.keys_read[bh] = kWindow + (int)kr;
        st[2] = found;
        st[3] = flags | kFlagDone;
        if (a.stats) {
          csa_head_stats hs = {found, kWindow + (int)kr, vr, (int)a.ncand[bh], 0, J, round + 1, 0};
          a.stats[bh] = hs;
        }
      }
    }
    __syncthreads();
  }
  if (found < 0 && tid == 0) {
    if (hi >= J) {
      // no certified level on the grid: exact attention (dense pass)
      a.beta[bh] = 0.f;
      a.level[bh] = J + 1;
      a.keys_read[bh] = (int)n;
      st[2] = J + 1;
      st[3] = flags | kFlagDone | kFlagFallback;
      if (a.stats) {
        csa_head_stats hs = {J + 1, (int)n, (int)n, (int)a.ncand[bh], 0, J, round + 1, 0};
        a.stats[bh] = hs;
      }
    } else {
      int nh = (round == 0) ? hi + 2 * a.r : J;
      if (round >= 1) nh = J;
      st[0] = hi;
      st[1] = nh > J ? J : nh;
    }
  }
}

// --------------------------------------------------- near-threshold count

template <int G>
__global__ void __launch_bounds__(256) near_kernel(const SparseArgs a, const __grid_constant__ SeqArgs seq) {
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int64_t n = seq.n[b];
  if (n <= kWindow || !a.stats) return;
  const int64_t P = n - kWindow;
  const int64_t key = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (key >= P) return;
  const int bh0 = b * a.Hq + g * G;
  const float* sp = a.s32 + ((int64_t)bg * a.pcap + key) * G;
  const float t = perturb_t(group_key(seq.seed[b], g), key);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int js = a.state[(int64_t)(bh0 + h) * 4 + 2];
    if (js < 0 || js > seq.J[b]) continue;
    const float s = sp[h];
    if (!(s > -INFINITY)) continue;
    const float dl = fsub(s, cmax_get(a, bh0 + h, 3));
    const float thr = -((float)js / (float)a.r) * 0.69314718f;
    const float x = dl + t * 0.69314718f;
    if (fabsf(x - thr) < 1e-5f || fabsf(dl - thr) < 1e-5f)
      atomicAdd(&a.stats[bh0 + h].n_near_threshold, 1);
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

cudaError_t launch_cstar(const SparseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, int64_t nmax_live,
                         cudaStream_t st) {
  dim3 grid((unsigned)((nmax_live + kTile - 1) / kTile), (unsigned)(a.B * a.Hkv));
  CSA_DG_SWITCH(cstar_kernel, <<<grid, 256, 0, st>>>(a, seq))
  return cudaGetLastError();
}
cudaError_t launch_rescore(const SparseArgs& a, const SeqArgs& seq, int d, int G, bool bf16,
                           int64_t pmax_live, cudaStream_t st) {
  dim3 grid((unsigned)((pmax_live + kTile - 1) / kTile), (unsigned)(a.B * a.Hkv));
  CSA_DG_SWITCH(rescore_kernel, <<<grid, 256, 0, st>>>(a, seq))
  return cudaGetLastError();
}
cudaError_t launch_predict(const SparseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, cudaStream_t st) {
  dim3 grid((unsigned)(a.B * a.Hkv));
  CSA_DG_SWITCH(predict_kernel, <<<grid, 256, 0, st>>>(a, seq))
  return cudaGetLastError();
}
cudaError_t launch_round(const SparseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, int64_t pmax_live,
                         int round, int nsm, cudaStream_t st) {
  dim3 grid((unsigned)((pmax_live + kTile - 1) / kTile), (unsigned)(a.B * a.Hkv));
  switch (G) {
    case 1: levels_kernel<1><<<grid, 256, 0, st>>>(a, seq); break;
    case 2: levels_kernel<2><<<grid, 256, 0, st>>>(a, seq); break;
    case 4: levels_kernel<4><<<grid, 256, 0, st>>>(a, seq); break;
    case 8: levels_kernel<8><<<grid, 256, 0, st>>>(a, seq); break;
    default: return cudaErrorInvalidValue;
  }
  const int nent = a.B * a.Hkv * a.J1;
  vplan_kernel<<<1, 1024, 0, st>>>(a, nent);
  dim3 vg((unsigned)(nsm * 4));
  CSA_DG_SWITCH(vgather_kernel, <<<vg, 256, 0, st>>>(a, seq, nent))
  dim3 cg((unsigned)(a.B * a.Hq));
  if (d == 128) certify_kernel<128><<<cg, 256, 0, st>>>(a, seq, round);
  else certify_kernel<64><<<cg, 256, 0, st>>>(a, seq, round);
  return cudaGetLastError();
}
cudaError_t launch_near(const SparseArgs& a, const SeqArgs& seq, int G, int64_t pmax_live, cudaStream_t st) {
  dim3 grid((unsigned)((pmax_live + 255) / 256), (unsigned)(a.B * a.Hkv));
  switch (G) {
    case 1: near_kernel<1><<<grid, 256, 0, st>>>(a, seq); break;
    case 2: near_kernel<2><<<grid, 256, 0, st>>>(a, seq); break;
    case 4: near_kernel<4><<<grid, 256, 0, st>>>(a, seq); break;
    case 8: near_kernel<8><<<grid, 256, 0, st>>>(a, seq); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace csa
