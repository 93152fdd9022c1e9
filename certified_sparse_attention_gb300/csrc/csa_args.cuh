// Argument blocks of the kernels and the launch functions of each
// translation unit (one definition, shared by the host layer).
#pragma once

#include <cuda.h>

#include "csa_internal.cuh"

namespace csa {

struct ScanArgs {
  const SeqArgs* seqd;    // per-sequence data in device memory (device-length
                          // steps), else null: the launch argument holds it
  const void* q;
  const uint8_t* K4;
  const float* bounds;
  float* ubar;          // [B*Hkv][n_max][G]
  float* hw;            // [B*Hkv][nblk_max][G] half width (ubar - l) / 2 per block
  float* tmax;          // [B*Hkv][ntile_max][G] largest ubar of each 256-key tile
  unsigned* cmax;       // [B*Hq][4] ordered floats: c_lo, c_hi, cb, c32
  unsigned* status;
  int Hq, Hkv;
  int64_t n_max, nblk_max;
  float rs;             // float32(1/sqrt d)
  bool two_digit;       // query codes of two s8 digits (QM = 127 * 257)
  // fused re-quantisation (device-length steps): the CTA whose tile holds
  // the block of token n - 1 rebuilds that block's codes, bounds, vmax and
  // vnorm2 from K and V before it scans it (the arrays it writes are named
  // in the ReqPtrs that follow *seqd in the workspace; a larger argument
  // block would cost the plain scan registers)
  bool requant;
  bool dp4a;            // integer dots by CUDA-core dp4a instead of tensor cores
};

// Arrays of the fused re-quantisation, stored right after the device-side
// SeqArgs of a device-length step.
struct ReqPtrs {
  const void* K;
  const void* V;
  uint8_t* K4;
  float* bounds;
  float* vmax;
  float* vnorm2;
};

struct SparseArgs {
  const SeqArgs* seqd;    // per-sequence data in device memory (device-length
                          // steps), else null: the launch argument holds it
  const void* q;
  const void* K;
  const void* V;
  const float* vmax;      // [B*Hkv][nblk_max]
  const float* vnorm2;    // [B*Hkv][n_max]        ||v_i||^2 per token
  const float* ubar;      // [B*Hkv][n_max][G]
  const float* hw;        // [B*Hkv][nblk_max][G] half width of the score bound per block
  const float* tmax;      // [B*Hkv][ntile_max][G] largest ubar of each 256-key tile
  float* s32;             // [B*Hkv][pcap][G]     scores (-inf: not a candidate, or not rescored)
  float* win;             // [B*Hkv][64][G]       window scores
  unsigned* cmax;         // [B*Hq][4]            c_lo, c_hi, cb, c32 (ordered)
  unsigned* jr_hist;      // [B*Hq][J1+1]         first level a key's K row is needed
  unsigned* ncand;        // [B*Hq]
  float* pre_hist;        // [B*Hq][J1][4]        d k, d D_B (value free, estimated); 2 unused
  float* acc;             // [B*Hq][J1][ACC]      d S1[D], d N_B[D], d k, d S2, d D_B, d H_B, d sampled
  float* winstats;        // [B*Hq][D+4]          N_R[D], D_R, H_R
  float* vmaxp;           // [B*Hkv]              max vmax over pool blocks
  int* state;             // [B*Hq][4]            lo, hi, stop, flags
  float* t32;             // [B*Hkv][pcap]([G])   perturbation t_i = -log2 u_i (per head if per_head)
  // 8-bit refinement tier (refine8 != 0)
  const uint8_t* K8;      // [B*Hkv][nblk_max*64][D] 8-bit codes
  const float* delta8;    // [B*Hkv][nblk_max][D]
  const float* bounds;    // [B*Hkv][nblk_max][2][D] (the minima m_c)
  uint16_t* jkey;         // [B*Hkv][pcap] per pool key: smallest bound level over the heads that
                          // can still need its row (bits 0-8; 0x1FF none), refined (bit 9),
                          // in the exact-max set (bit 10)
  int* jrd;               // [B*Hq][J1+1] keys_read histogram moves of the refinement
  uint16_t* jref;         // [B*Hkv][pcap][G] refined level of a refined key per head (diagnostics)
  unsigned* ninset;       // [B*Hq] pool keys in the head's exact-max set
  int refine8;            // 0 off, 1 every group, 2 groups whose first range reaches level r
  float* pref;            // [B*Hq][ACC]          a continuing head's sums through its last range
  uint2* xlist;           // [B*Hkv][n_max]       exact-max set: key, head mask
  unsigned* xcnt;         // [B*Hkv]
  unsigned* chunk_map;    // [nchunk_cap]         gather work item -> bucket entry
  int64_t nchunk_cap;
  uint2* clist;           // [B*Hkv][pcap]        candidates: key, head mask | min bound level << 8
  int* front;             // [4][B*Hkv]           rescored through bound level (+1) before round r
  unsigned* ccnt;         // [B*Hkv]
  unsigned* nfall;        // heads that need the exact fallback
  unsigned* rq;           // round queues: [3][B*Hkv] groups per round, [3][B*Hkv] flags,
                          // [3] group counts, [3] work-item counters
  unsigned* bcnt;         // [3][B*Hkv][J1]        entries appended in each round
  unsigned* bcons;        // [B*Hkv][J1]           entries over the step (diagnostics)
  uint2* buckets;         // [B*Hkv][J1][pcap]    key, event masks (add | trans<<8 | before<<16)
  unsigned* plan_start;   // [B*Hkv*J1]
  unsigned* plan_end;     // [B*Hkv*J1]
  unsigned* plan_off;     // [B*Hkv*J1 + 1]
  unsigned* status;
  float* o;
  float* beta;
  int* level;
  int* keys_read;
  csa_head_stats* stats;
  int B, Hq, Hkv;
  int64_t n_max, nblk_max, pcap;
  int J1;                 // level stride: largest J + 1
  int r;
  float eps, delta;
  int measure;
  int per_head;           // one perturbation draw per query head
  float zclt;             // two-sided normal quantile at delta (CLT rule)
  float rs;               // float32(1/sqrt d)
};

struct DenseArgs {
  const SeqArgs* seqd;    // per-sequence data in device memory (device-length
                          // steps), else null: the launch argument holds it
  const void* q;
  const void* K;
  const void* V;
  float* part;            // [nsplit][B*Hq][D+2]: m, l, acc[D]
  float* o;               // [B*Hq][D]
  const int* state;       // optional [B*Hq][4]: only heads with flag bit 0
  const unsigned* nfall;  // optional: skip everything when it reads 0
  unsigned* status;       // optional: status word (bit 4: a bounded wait gave up)
  int B, Hq, Hkv;
  int64_t n_max;
  int nsplit;
  float rs;
};

struct QuantArgs {
  const SeqArgs* seqd;    // per-sequence data in device memory (device-length
                          // steps), else null: the launch argument holds it
  const void* K;
  const void* V;
  uint8_t* K4;
  float* bounds;
  float* vmax;
  float* vnorm2;
  uint8_t* K8;          // 8-bit codes [B*Hkv][nblk_max*64][D] (quant8_kernel)
  float* delta8;        // [B*Hkv][nblk_max][D]
  int Hkv;
  int64_t n_max, nblk_max;
  int64_t blk_from;
};

// tm_codes: a tensor map over the 4-bit code rows (make_tmap_2d_u8_sw64,
// box 64 bytes x 256 rows) for the plain d = 128 scan, or null (16-byte
// cp.async staging)
cudaError_t launch_scan(const ScanArgs&, const SeqArgs&, int B, int d, int G, bool bf16, int64_t nmax_live,
                        const CUtensorMap* tm_codes, cudaStream_t);
cudaError_t launch_cstar(const SparseArgs&, const SeqArgs&, int d, int G, bool bf16, int64_t nmax_live,
                         int nsm, cudaStream_t);
cudaError_t launch_candidates(const SparseArgs&, const SeqArgs&, int G, int64_t pmax_live, int nsm, cudaStream_t);
cudaError_t launch_predict(const SparseArgs&, const SeqArgs&, int d, int G, bool bf16, cudaStream_t);
typedef void (*PhaseMark)(int phase, cudaStream_t);
cudaError_t launch_round(const SparseArgs&, const SeqArgs&, int d, int G, bool bf16, int64_t pmax_live,
                         int round, int nsm, cudaStream_t, PhaseMark mark);
cudaError_t launch_near(const SparseArgs&, const SeqArgs&, int G, int64_t pmax_live, cudaStream_t);
cudaError_t launch_dense(const DenseArgs&, const SeqArgs&, int d, int G, bool bf16, int64_t nmax_live,
                         cudaStream_t);
cudaError_t launch_quant(const QuantArgs&, const SeqArgs&, int B, int d, bool bf16, int64_t nblocks,
                         cudaStream_t);
cudaError_t launch_quant8(const QuantArgs&, const SeqArgs&, int B, int d, bool bf16, int64_t nblocks,
                          cudaStream_t);
int dense_nsplit(int64_t n_max);
cudaError_t launch_seq_prep(const int64_t* len, const uint64_t* seed, int B, int64_t n_max, int r, int J_override,
                            SeqArgs* out, const ReqPtrs& req, unsigned* status, cudaStream_t);

// Launch with programmatic stream serialisation (see pdl_entry).
template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, args...);
}
void add_launches(int k);   // adds to the launch count csa_profile_read reports

// Unique id of the calling thread's current CUDA context (the driver's
// cuCtxGetId, reached through the runtime's driver entry points, so that the
// library does not link libcuda).  Returns false when no context is current.
// Per-device state tied to a context (a device address of a file-scope
// array, library streams) is keyed on this id: after a device reset the
// runtime creates a new primary context, with a new id.
bool current_context_id(unsigned long long* id);

// A 2-D tensor map over a row-major array of `rows` rows of `inner` 16-bit
// elements (row pitch `pitch_bytes`), box = box_inner x box_rows elements,
// 128-byte swizzle, zero fill out of bounds (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry points).  False if the driver refuses
// (base or pitch not 16-byte aligned, sizes out of range).
bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                       uint32_t box_inner, uint32_t box_rows);
// The same over `rows` rows of `inner` bytes (8-bit elements), 64-byte
// swizzle (the 16-byte chunk c of tile row r lands at chunk c ^ ((r / 2) % 4)
// of a 512-byte-aligned buffer).
bool make_tmap_2d_u8_sw64(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                          uint32_t box_inner, uint32_t box_rows);

}  // namespace csa
