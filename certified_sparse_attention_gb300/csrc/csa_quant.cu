// 4-bit per-block, per-channel key quantiser and per-block value-norm bound.
//
// picx.dev summary, "Algorithm Components" 4: keys quantised to 4 bits per
// block and channel, the KIVI scheme.  Per 64-token block (aligned to
// position 0, the tokens present only) and channel c:
//   m_c = min, Delta_c = fl((max - min) / 15) (0 -> 1),
//   code = clamp(rint(fl(fl(k - m_c) / Delta_c)), 0, 15)   (ties to even),
// two codes per byte with the even channel in the low nibble.  vmax of the
// block = max over its tokens of sqrt(sequential float32 sum of v_c^2),
// times (1 + 2^-16), an upper bound on every ||v_i|| of the block; the sums
// themselves are kept per token (vnorm2) for the value gather.
// One CTA per (sequence, KV head, block); thread c owns channel c.
#include "csa_args.cuh"

namespace csa {

template <int D, typename E>
__global__ void __launch_bounds__(D) quant_kernel(const QuantArgs a, const __grid_constant__ SeqArgs seq) {
  pdl_entry();
  __shared__ float s_vm[kBlock];
  const int c = threadIdx.x;
  const int bg = blockIdx.y, b = bg / a.Hkv;
  const int64_t n = seq.n[b];
  const int64_t blk = a.blk_from + blockIdx.x;
  const int64_t t0 = blk * kBlock;
  if (t0 >= n) return;
  const int rows = (int)min((int64_t)kBlock, n - t0);
  const E* Kb = reinterpret_cast<const E*>(a.K) + ((int64_t)bg * a.n_max + t0) * D;
  const E* Vb = reinterpret_cast<const E*>(a.V) + ((int64_t)bg * a.n_max + t0) * D;
  float mn = INFINITY, mx = -INFINITY;
  for (int t = 0; t < rows; ++t) {
    const float k = Elem<E>::get(Kb, (int64_t)t * D + c);
    mn = fminf(mn, k);
    mx = fmaxf(mx, k);
  }
  float dl = fdiv(fsub(mx, mn), 15.0f);
  if (dl == 0.0f) dl = 1.0f;
  float* bp = a.bounds + ((int64_t)bg * a.nblk_max + blk) * 2 * D;
  bp[c] = mn;
  bp[D + c] = dl;
  uint8_t* kp = a.K4 + ((int64_t)bg * a.nblk_max * kBlock + t0) * (D / 2);
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
    if (t0 + c < a.n_max) a.vnorm2[(int64_t)bg * a.n_max + t0 + c] = ss;
  }
  __syncthreads();
  if (c == 0) {
    float m = 0.0f;
    for (int t = 0; t < rows; ++t) m = fmaxf(m, s_vm[t]);
    a.vmax[(int64_t)bg * a.nblk_max + blk] = fmul(m, 1.0000152587890625f);
  }
}

cudaError_t launch_quant(const QuantArgs& a, const SeqArgs& seq, int B, int d, bool bf16, int64_t nblocks,
                         cudaStream_t st) {
  if (nblocks <= 0) return cudaSuccess;
  dim3 grid((unsigned)nblocks, (unsigned)(B * a.Hkv));
  if (d == 128) {
    if (bf16) launch_pdl(quant_kernel<128, __nv_bfloat16>, grid, dim3(128), 0, st, a, seq);
    else launch_pdl(quant_kernel<128, float>, grid, dim3(128), 0, st, a, seq);
  } else {
    if (bf16) launch_pdl(quant_kernel<64, __nv_bfloat16>, grid, dim3(64), 0, st, a, seq);
    else launch_pdl(quant_kernel<64, float>, grid, dim3(64), 0, st, a, seq);
  }
  return cudaGetLastError();
}

}  // namespace csa
