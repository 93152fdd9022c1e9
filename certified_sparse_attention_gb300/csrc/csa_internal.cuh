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
#ifndef CSA_CAND_SEG
#define CSA_CAND_SEG 3072
#endif
// pool keys per candidate-list segment (one candidate CTA).  On the 128K x 4
// step with two sub-batch chains: 2048, 2560, 3072, 3584 and 4096 keys gave
// 655, 645, 640, 648 and 658 us (the unsplit candidate pass alone is
// fastest at 2048: 102 against 109 us).
constexpr int kCandSeg = CSA_CAND_SEG;
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

// --------------------------------------------- bulk tensor copies (TMA)
//
// Tiles move from global to shared memory with cp.async.bulk.tensor (the
// tensor memory accelerator), completing on an mbarrier with a transaction
// byte count.  Every wait on an mbarrier is bounded in time: after
// kWaitNs nanoseconds it gives up and returns false, the caller records
// CSA_ERR_TIMEOUT in the status word and leaves.

constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
// make initialised barriers visible to the async proxy (the copies)
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(unsigned bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// wait for the phase of parity `parity` to complete; false after kWaitNs
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity) {
  unsigned long long t0 = 0;
  for (unsigned it = 0;; ++it) {
    unsigned done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if (it == 0) t0 = global_ns();
    else if ((it & 63u) == 0u && global_ns() - t0 > kWaitNs) return false;
  }
}
// 2-D tiled load of box (x, y) of `map` into shared memory at dst
__device__ __forceinline__ void tma_load_2d(unsigned dst, const void* map, int x, int y, unsigned bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];\n" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// barrier over the first `count` threads of the CTA (named barrier `id`)
__device__ __forceinline__ void bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// ------------------------------------------------------ block quantiser
//
// 4-bit per-block, per-channel key codes and the block's value-norm data
// (picx.dev "Algorithm Components" 4, the KIVI scheme).  For the 64-token
// block `blk` of group bg (aligned to position 0; tokens present: those
// below n) and channel c:
//   m_c = min, Delta_c = fl((max - min) / 15) (0 -> 1),
//   code = clamp(rint(fl(fl(k - m_c) / Delta_c)), 0, 15)   (ties to even),
// two codes per byte with the even channel in the low nibble (positions of
// the block at or past n get code 0 and vnorm2 0).  vnorm2 of a token is
// the sequential float32 sum of v_c^2; vmax of the block = max over its
// tokens of sqrt(vnorm2), times (1 + 2^-16): an upper bound on every
// ||v_i|| of the block.  Thread c < D owns channel c; every thread of the
// CTA calls it (it holds a barrier).
template <int D, typename E>
__device__ __forceinline__ void quantize_block(const void* K, const void* V, uint8_t* K4, float* bounds,
                                               float* vmax, float* vnorm2, int64_t n_max, int64_t nblk_max,
                                               int bg, int64_t blk, int64_t n, float* s_vm) {
  const int c = threadIdx.x;
  const int64_t t0 = blk * kBlock;
  const int rows = (int)min((int64_t)kBlock, n - t0);
  const E* Kb = reinterpret_cast<const E*>(K) + ((int64_t)bg * n_max + t0) * D;
  const E* Vb = reinterpret_cast<const E*>(V) + ((int64_t)bg * n_max + t0) * D;
  if (c < D) {
    float mn = INFINITY, mx = -INFINITY;
    for (int t = 0; t < rows; ++t) {
      const float k = Elem<E>::get(Kb, (int64_t)t * D + c);
      mn = fminf(mn, k);
      mx = fmaxf(mx, k);
    }
    float dl = fdiv(fsub(mx, mn), 15.0f);
    if (dl == 0.0f) dl = 1.0f;
    float* bp = bounds + ((int64_t)bg * nblk_max + blk) * 2 * D;
    bp[c] = mn;
    bp[D + c] = dl;
    uint8_t* kp = K4 + ((int64_t)bg * nblk_max * kBlock + t0) * (D / 2);
    for (int t = 0; t < kBlock; ++t) {
      int code = 0;
      if (t < rows) {
        const float k = Elem<E>::get(Kb, (int64_t)t * D + c);
        float x = rintf(fdiv(fsub(k, mn), dl));
        x = fminf(fmaxf(x, 0.0f), 15.0f);
        code = (int)x;
      }
      const int hi = __shfl_down_sync(0xffffffffu, code, 1);
      if ((c & 1) == 0) kp[(int64_t)t * (D / 2) + c / 2] = (uint8_t)(code | (hi << 4));
    }
  }
  // value norms: thread t < rows walks its row sequentially
  if (c < kBlock) {
    float nrm = 0.0f, ss = 0.0f;
    if (c < rows) {
      for (int x = 0; x < D; ++x) {
        const float v = Elem<E>::get(Vb, (int64_t)c * D + x);
        ss = fadd(ss, fmul(v, v));
      }
      nrm = __fsqrt_rn(ss);
    }
    s_vm[c] = nrm;
    if (t0 + c < n_max) vnorm2[(int64_t)bg * n_max + t0 + c] = ss;
  }
  __syncthreads();
  if (c == 0) {
    float m = 0.0f;
    for (int t = 0; t < rows; ++t) m = fmaxf(m, s_vm[t]);
    vmax[(int64_t)bg * nblk_max + blk] = fmul(m, 1.0000152587890625f);
  }
}

// 8-bit codes of the same blocks for the refinement tier (picx.dev
// "Algorithm Components" 4: an 8-bit stage between the 4-bit candidates and
// the exact 16-bit reads): per block and channel the same minimum m_c,
// Delta8_c = fl((max - min) / 255) (0 -> 1),
// code = clamp(rint(fl(fl(k - m_c) / Delta8_c)), 0, 255); one byte per code,
// positions at or past n get code 0.  Thread c < D owns channel c.
template <int D, typename E>
__device__ __forceinline__ void quantize_block8(const void* K, uint8_t* K8, float* delta8, int64_t n_max,
                                                int64_t nblk_max, int bg, int64_t blk, int64_t n) {
  const int c = threadIdx.x;
  if (c >= D) return;
  const int64_t t0 = blk * kBlock;
  const int rows = (int)min((int64_t)kBlock, n - t0);
  const E* Kb = reinterpret_cast<const E*>(K) + ((int64_t)bg * n_max + t0) * D;
  float mn = INFINITY, mx = -INFINITY;
  for (int t = 0; t < rows; ++t) {
    const float k = Elem<E>::get(Kb, (int64_t)t * D + c);
    mn = fminf(mn, k);
    mx = fmaxf(mx, k);
  }
  float dl = fdiv(fsub(mx, mn), 255.0f);
  if (dl == 0.0f) dl = 1.0f;
  delta8[((int64_t)bg * nblk_max + blk) * D + c] = dl;
  uint8_t* kp = K8 + ((int64_t)bg * nblk_max * kBlock + t0) * D;
  for (int t = 0; t < kBlock; ++t) {
    int code = 0;
    if (t < rows) {
      const float k = Elem<E>::get(Kb, (int64_t)t * D + c);
      float x = rintf(fdiv(fsub(k, mn), dl));
      x = fminf(fmaxf(x, 0.0f), 255.0f);
      code = (int)x;
    }
    kp[(int64_t)t * D + c] = (uint8_t)code;
  }
}

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
