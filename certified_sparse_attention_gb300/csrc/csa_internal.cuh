// Device helpers shared by the kernels of the library.
//
// The float32 sequences below are the fixed operation orders that make the
// 4-bit bounds, the perturbations and the candidate levels reproducible bit
// for bit: every add / multiply / divide is an explicitly rounded
// (__fadd_rn, __fmul_rn, __fdiv_rn) IEEE binary32 operation, never fused.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/csa.h"

namespace csa {

constexpr int kBlock = 64;     // quantisation block (tokens)
constexpr int kWindow = 64;    // window read exactly (last tokens)
constexpr int kTile = 256;     // keys per scan / candidate tile
constexpr int kCandSeg = 4096; // pool keys per candidate-list segment (one candidate CTA)
constexpr int kMaxB = 128;     // sequences per call
constexpr int kMaxHeads = 1024; // query heads and KV heads per call
constexpr int kMaxJ = 255;     // last grid level supported
constexpr int kMaxSub = 4;     // sub-batches of one decode call
constexpr int kHeadStream = 1 << 20;   // stream ids of per-query-head draws start here

// Per-call sequence data passed by value (graph-capturable).
struct SeqArgs {
  int64_t n[kMaxB];
  unsigned long long seed[kMaxB];
  int J[kMaxB];          // last grid level of each sequence
};

// ---------------------------------------------------------------- floats

__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fdiv(float a, float b) { return __fdiv_rn(a, b); }

// float32(1 / ln 2)
__device__ __forceinline__ float log2e_f() { return __int_as_float(0x3FB8AA3B); }

// Monotone map float -> uint for atomicMax on floats (0 is below every
// mapped value, so a zeroed slot means "no value yet").
__device__ __forceinline__ unsigned ord_of(float f) {
  unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_of_ord(unsigned o) {
  unsigned u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}
__device__ __forceinline__ void atomic_max_f(unsigned* slot, float v) {
  atomicMax(slot, ord_of(v));
}

// ------------------------------------------------------------ element I/O

template <typename E> struct Elem;
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float get(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
  }
  // four consecutive elements (8-byte aligned)
  static __device__ __forceinline__ float4 get4(const __nv_bfloat16* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    float4 f;
    f.x = __uint_as_float(u.x << 16);
    f.y = __uint_as_float(u.x & 0xFFFF0000u);
    f.z = __uint_as_float(u.y << 16);
    f.w = __uint_as_float(u.y & 0xFFFF0000u);
    return f;
  }
  static __device__ __forceinline__ float2 get2(const __nv_bfloat16* p) {
    unsigned u = *reinterpret_cast<const unsigned*>(p);
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  }
};
template <> struct Elem<float> {
  static __device__ __forceinline__ float get(const float* p, int64_t i) { return p[i]; }
  static __device__ __forceinline__ float4 get4(const float* p) {
    return *reinterpret_cast<const float4*>(p);
  }
  static __device__ __forceinline__ float2 get2(const float* p) {
    return *reinterpret_cast<const float2*>(p);
  }
};

// ---------------------------------------------------------- perturbations
// SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): the k-th output of a
// generator seeded with s is mix64(s + k * gamma).

constexpr unsigned long long kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Group key for (sequence seed, KV head g).
__device__ __forceinline__ unsigned long long group_key(unsigned long long seed, int g) {
  return mix64(seed + (unsigned long long)(g + 1) * kGamma);
}

// log2(m) for integers m in [1, 2^53], float32.  Exponent from the bit
// length; the top 24 bits of m as the mantissa f in [1, 2) (truncation);
// f > sqrt2 halved; log f = 2 atanh(z), z = (f-1)/(f+1), series through z^9
// (Abramowitz & Stegun 4.1.27), Horner in z^2.
__device__ __forceinline__ float log2_m53(unsigned long long m) {
  int e = 63 - __clzll((long long)m);
  int sh = e > 23 ? e - 23 : 0;
  unsigned top = (unsigned)(m >> sh);                  // < 2^24: exact
  int k = e - sh;                                      // 0..23
  float f = fmul(__uint2float_rn(top), __int_as_float((127 - k) << 23));
  if (f > __int_as_float(0x3FB504F3)) {                // float32(sqrt 2)
    f = fmul(f, 0.5f);
    e += 1;
  }
  float z = fdiv(fsub(f, 1.0f), fadd(f, 1.0f));
  float z2 = fmul(z, z);
  float p = fmul(__int_as_float(0x3DE38E39), z2);     // float32(1/9)
  p = fadd(p, __int_as_float(0x3E124925));            // float32(1/7)
  p = fmul(p, z2);
  p = fadd(p, __int_as_float(0x3E4CCCCD));            // float32(1/5)
  p = fmul(p, z2);
  p = fadd(p, __int_as_float(0x3EAAAAAB));            // float32(1/3)
  p = fmul(p, z2);
  p = fadd(p, 1.0f);
  float l2f = fmul(fmul(z, p), __int_as_float(0x4038AA3B));   // float32(2/ln2)
  return fadd((float)e, l2f);
}

// t_i = -log2 u_i with u_i = ((h_i >> 11) + 1) 2^-53, h_i the (i+1)-th
// output of the group's generator.
__device__ __forceinline__ float perturb_t(unsigned long long gkey, long long i) {
  unsigned long long h = mix64(gkey + (unsigned long long)(i + 1) * kGamma);
  unsigned long long m = (h >> 11) + 1ull;
  return fsub(53.0f, log2_m53(m));
}

// ----------------------------------------------------------------- levels

// max(0, ceil(v)) with everything above J (and NaN) mapped to J + 1.
__device__ __forceinline__ int level_of(float v, int J) {
  if (!(v <= (float)J)) return J + 1;
  if (v <= 0.0f) return 0;
  return (int)ceilf(v);
}

// Bound level jbar from the 4-bit upper bound ub, the certified lower bound
// cb of the maximum score and the perturbation t:
//   xbar = fl(fl(fl(ub - cb) * log2e) + t),  jbar = ceil(fl(fl(-r xbar) - 2^-10)).
__device__ __forceinline__ int bound_level(float ub, float cb, float t, float neg_r, int J) {
  float xb = fadd(fmul(fsub(ub, cb), log2e_f()), t);
  float y = fsub(fmul(neg_r, xb), 0.0009765625f);
  return level_of(y, J);
}

// Exact inclusion level j and heavy level h from the float32 score s and the
// float32 maximum c (sampled at level j' iff j <= j'; heavy iff h <= j').
__device__ __forceinline__ void exact_levels(float s, float c, float t, float neg_r, int J,
                                             int& jl, int& hl) {
  float y = fmul(fsub(s, c), log2e_f());
  float x = fadd(y, t);
  jl = level_of(fmul(neg_r, x), J);
  hl = level_of(fmul(neg_r, y), J);
}

// ------------------------------------------ programmatic dependent launch
//
// Every kernel of the library is launched with programmatic stream
// serialisation (launch_pdl): the next kernel on the stream may be
// scheduled while this one's last CTAs run.  Each kernel therefore starts
// by waiting for its predecessor grid (its results are then visible), and
// then lets its own dependent launch.
__device__ __forceinline__ void pdl_entry() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ------------------------------------------------------- async staging

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
  int src = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sa), "l"(gmem), "r"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ------------------------------------------------------ warp row products
//
// Eight rows at a time: lane l holds channels [l*CPL, (l+1)*CPL) of every
// row (CPL = D/32).  part[r] is the lane's float32 partial of row r.  After
// the call lane l holds in part[0] the full sum of row (l & 7).  The sum is
// the adjacent-pair tree over the lanes (pairs l, l^1 first, then l^2, ...),
// which together with the lane-local tree is the adjacent-pair tree over
// the D channels.
__device__ __forceinline__ float reduce8_rows(float part[8]) {
  const int lane = threadIdx.x & 31;
  // stage over lane bit 0: keep rows whose bit 0 equals the lane's
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    bool hi = lane & 1;
    float send = hi ? part[2 * i] : part[2 * i + 1];
    float keep = hi ? part[2 * i + 1] : part[2 * i];
    float got = __shfl_xor_sync(0xffffffffu, send, 1);
    part[i] = fadd(keep, got);
  }
  // now part[i] is row (2i + bit0); stage over lane bit 1
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    bool hi = (lane >> 1) & 1;
    float send = hi ? part[2 * i] : part[2 * i + 1];
    float keep = hi ? part[2 * i + 1] : part[2 * i];
    float got = __shfl_xor_sync(0xffffffffu, send, 2);
    part[i] = fadd(keep, got);
  }
  // part[i] is row (4i + 2 bit1 + bit0); stage over lane bit 2
  {
    bool hi = (lane >> 2) & 1;
    float send = hi ? part[0] : part[1];
    float keep = hi ? part[1] : part[0];
    float got = __shfl_xor_sync(0xffffffffu, send, 4);
    part[0] = fadd(keep, got);
  }
  float v = part[0];
  v = fadd(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fadd(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}

// Lane-local adjacent-pair tree over CPL products (CPL = 2 or 4).
template <int CPL>
__device__ __forceinline__ float local_tree(const float* p) {
  if (CPL == 2) return fadd(p[0], p[1]);
  return fadd(fadd(p[0], p[1]), fadd(p[2], p[3]));
}

}  // namespace csa
