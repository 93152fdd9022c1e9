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
__global__ void __launch_bounds__(256) dense_split_kernel(const DenseArgs a, const __grid_constant__ SeqArgs seq,
                                                          int nsplit_live) {
  pdl_entry();
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
__global__ void __launch_bounds__(128) dense_combine_kernel(const DenseArgs a, const __grid_constant__ SeqArgs seq) {
  pdl_entry();
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

cudaError_t launch_dense(const DenseArgs& a, const SeqArgs& seq, int d, int G, bool bf16, int64_t nmax_live,
                         cudaStream_t st) {
  const int nsplit_live = (int)((nmax_live + kDenseChunk - 1) / kDenseChunk);
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
