// Dense decode attention with its split-K partials in a fixed, file-scope
// device array instead of a caller-supplied workspace: the library's one
// entry point that needs no device allocation by anyone.  It exists for
// callers that cannot allocate device memory at the point of the call: a
// plain C host program that links only this library and owns no device
// allocator, or a callback that runs while another component holds all of
// the device memory and its allocator's lock.  The kernels are the same two
// launches csa_dense_decode makes; only where the partials live differs.
#include <cmath>
#include <cstring>
#include <mutex>

#include "csa_args.cuh"

namespace csa {

namespace {

constexpr size_t kStaticScratchBytes = (size_t)CSA_DENSE_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// Split-K partials, [nsplit][B*Hq][d+2] floats.  Every slot the combine
// kernel reads is written by the split kernel of the same call first, so the
// contents on entry do not matter and nothing has to start at zero.  One
// array per device, shared by every call on that device: two calls whose
// kernels overlap in time (different streams, or host threads) race on it.
static __device__ __align__(256) unsigned char g_dense_scratch[kStaticScratchBytes];

std::mutex g_addr_mu;
struct ScratchAddr {
  void* ptr;
  unsigned long long ctx;   // context the address belongs to
};
ScratchAddr g_addr[kMaxDevices] = {};

// Device address of g_dense_scratch in the current device's context.  The
// host-side name g_dense_scratch is only a stand-in for the array (a kernel
// given it would fault, or where the GPU can reach host memory, quietly use
// the wrong memory); the device address comes from cudaGetSymbolAddress,
// made with the device current.  A call made outside a stream capture looks
// it up every time (cheap once the module is loaded; the first lookup on a
// device loads the module) and caches it with the context's id; a call
// inside a capture takes the cached address of its device and context, and
// fails if there is none.  So a device reset, which ends the context and
// the module holding the array, can never leave a stale address in use.
csa_status scratch_address(cudaStream_t st, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return CSA_ERR_CUDA;
  if (dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) return CSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_addr_mu);
  unsigned long long ctx = 0;
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    // also makes the device's primary context current if it was not
    if (cudaGetSymbolAddress(&p, g_dense_scratch) != cudaSuccess || !p) return CSA_ERR_CUDA;
    if (!current_context_id(&ctx)) return CSA_ERR_CUDA;
    g_addr[dev].ptr = p;
    g_addr[dev].ctx = ctx;
  } else if (!current_context_id(&ctx) || !g_addr[dev].ptr || g_addr[dev].ctx != ctx) {
    return CSA_ERR_CUDA;   // no lookup made outside a capture in this context
  }
  *out = g_addr[dev].ptr;
  return CSA_OK;
}

}  // namespace
}  // namespace csa

using namespace csa;

extern "C" {

csa_status csa_dense_decode_static(const csa_shape* shape, const void* q, const void* K, const void* V,
                                   const int64_t* len, float* o, void* stream) {
  if (!shape || !q || !K || !V || !len || !o) return CSA_ERR_INVALID_ARG;
  const size_t need = csa_dense_workspace_size(shape);
  if (need == 0) {
    // invalid or unsupported shape: report which, as csa_dense_decode does
    const bool valid = shape->B >= 1 && shape->Hq >= 1 && shape->Hkv >= 1 && shape->Hq <= kMaxHeads &&
                       shape->Hkv <= kMaxHeads && shape->Hq % shape->Hkv == 0 &&
                       shape->n_max >= 1 && shape->n_max <= (int64_t)1 << 31 &&
                       (shape->dtype == CSA_BF16 || shape->dtype == CSA_F32);
    return valid ? CSA_ERR_UNSUPPORTED : CSA_ERR_INVALID_ARG;
  }
  if (need > kStaticScratchBytes) return CSA_ERR_WORKSPACE;
  SeqArgs seq;
  std::memset(&seq, 0, sizeof(seq));
  int64_t nlive = 0;
  for (int b = 0; b < shape->B; ++b) {
    if (len[b] < 1 || len[b] > shape->n_max) return CSA_ERR_INVALID_ARG;
    seq.n[b] = len[b];
    if (len[b] > nlive) nlive = len[b];
  }
  void* scratch = nullptr;
  const csa_status sa = scratch_address((cudaStream_t)stream, &scratch);
  if (sa != CSA_OK) return sa;
  // the array holds the status word, then the partials (the workspace
  // layout of csa_dense_decode)
  if (cudaMemsetAsync(scratch, 0, sizeof(unsigned), (cudaStream_t)stream) != cudaSuccess) return CSA_ERR_CUDA;
  DenseArgs a = {};
  a.q = q; a.K = K; a.V = V; a.part = (float*)((char*)scratch + 256); a.o = o; a.state = nullptr;
  a.nfall = nullptr; a.status = (unsigned*)scratch;
  a.B = shape->B; a.Hq = shape->Hq; a.Hkv = shape->Hkv; a.n_max = shape->n_max;
  a.nsplit = dense_nsplit(shape->n_max); a.rs = (float)(1.0 / std::sqrt((double)shape->d));
  add_launches(2);
  return launch_dense(a, seq, shape->d, shape->Hq / shape->Hkv, shape->dtype == CSA_BF16, nlive,
                      (cudaStream_t)stream) == cudaSuccess
             ? CSA_OK
             : CSA_ERR_CUDA;
}

}  // extern "C"
