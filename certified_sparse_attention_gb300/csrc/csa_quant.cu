// Input preparation of the decode step.
//
// quant_kernel: the 4-bit per-block, per-channel key quantiser and the
// value-norm data (picx.dev summary, "Algorithm Components" 4: the KIVI
// scheme; the arithmetic is quantize_block in csa_internal.cuh), one CTA
// per (sequence, KV head, block) with thread c on channel c, for the
// blocks that hold a token at or past `from_token`.
// seq_prep_kernel: the per-sequence data of a step whose lengths and seeds
// are in device memory.
#include "csa_args.cuh"

namespace csa {

template <int D, typename E>
__global__ void __launch_bounds__(D) quant_kernel(const QuantArgs a, const __grid_constant__ SeqArgs seq_arg) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  __shared__ float s_vm[kBlock];
  const int bg = blockIdx.y, b = bg / a.Hkv;
  const int64_t n = seq.n[b];
  const int64_t blk = a.blk_from + blockIdx.x;
  if (blk * kBlock >= n) return;
  quantize_block<D, E>(a.K, a.V, a.K4, a.bounds, a.vmax, a.vnorm2, a.n_max, a.nblk_max, bg, blk, n, s_vm);
}

template <int D, typename E>
__global__ void __launch_bounds__(D) quant8_kernel(const QuantArgs a, const __grid_constant__ SeqArgs seq_arg) {
  pdl_entry();
  const SeqArgs& seq = a.seqd ? *a.seqd : seq_arg;
  const int bg = blockIdx.y, b = bg / a.Hkv;
  const int64_t n = seq.n[b];
  const int64_t blk = a.blk_from + blockIdx.x;
  if (blk * kBlock >= n) return;
  quantize_block8<D, E>(a.K, a.K8, a.delta8, a.n_max, a.nblk_max, bg, blk, n);
}

cudaError_t launch_quant8(const QuantArgs& a, const SeqArgs& seq, int B, int d, bool bf16, int64_t nblocks,
                          cudaStream_t st) {
  if (nblocks <= 0) return cudaSuccess;
  dim3 grid((unsigned)nblocks, (unsigned)(B * a.Hkv));
  if (d == 128) {
    if (bf16) launch_pdl(quant8_kernel<128, __nv_bfloat16>, grid, dim3(128), 0, st, a, seq);
    else launch_pdl(quant8_kernel<128, float>, grid, dim3(128), 0, st, a, seq);
  } else {
    if (bf16) launch_pdl(quant8_kernel<64, __nv_bfloat16>, grid, dim3(64), 0, st, a, seq);
    else launch_pdl(quant8_kernel<64, float>, grid, dim3(64), 0, st, a, seq);
  }
  return cudaGetLastError();
}

// Per-sequence data of a step whose lengths and seeds live in device
// memory: n, seed and the last grid level J = ceil(r log2 |pool|) (the
// smallest j with 2^j >= |pool|^r, in exact 128-bit integers), followed by
// the arrays of the fused re-quantisation.  A length outside [1, n_max] is
// clamped and flagged in the status word (bit 8).
__global__ void __launch_bounds__(kMaxB) seq_prep_kernel(const int64_t* len, const unsigned long long* seed, int B,
                                                       int64_t n_max, int r, int J_override, SeqArgs* out,
                                                       ReqPtrs req, unsigned* status) {
  pdl_entry();
  const int b = threadIdx.x;
  if (b == 0) *reinterpret_cast<ReqPtrs*>(out + 1) = req;
  if (b >= kMaxB) return;
  if (b >= B) {
    out->n[b] = 0; out->seed[b] = 0ull; out->J[b] = 0;
    return;
  }
  int64_t n = len[b];
  if (n < 1 || n > n_max) {
    atomicOr(status, 8u);
    n = n < 1 ? 1 : n_max;
  }
  const int64_t P = n > kWindow ? n - kWindow : 0;
  int J = 0;
  if (J_override >= 0) {
    J = J_override;
  } else if (P > 1) {
    unsigned __int128 t = 1;
    for (int i = 0; i < r; ++i) t *= (unsigned __int128)P;
    while ((((unsigned __int128)1) << J) < t) ++J;
  }
  out->n[b] = n;
  out->seed[b] = seed[b];
  out->J[b] = J;
}

cudaError_t launch_seq_prep(const int64_t* len, const uint64_t* seed, int B, int64_t n_max, int r, int J_override,
                            SeqArgs* out, const ReqPtrs& req, unsigned* status, cudaStream_t st) {
  launch_pdl(seq_prep_kernel, dim3(1), dim3(kMaxB), 0, st, len, (const unsigned long long*)seed, B, n_max, r,
             J_override, out, req, status);
  return cudaGetLastError();
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
