// Host side of the C ABI declared in include/csa.h: argument checks, the
// workspace layout, the exact grid size J = ceil(r log2 |pool|), and the
// launch sequence of one decode step.  No device memory is allocated here.
#include <algorithm>
#include <cmath>
#include <cuda.h>
#include <mutex>
#include <cstring>

#include "csa_args.cuh"

namespace csa {

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// J = smallest j with 2^j >= P^r (so tau_J = 2^(-j/r) <= 1/P); exact integers.
int grid_J(int64_t P, int r) {
  if (P <= 1) return 0;
  unsigned __int128 target = 1;
  for (int i = 0; i < r; ++i) target *= (unsigned __int128)P;
  int j = 0;
  while (((unsigned __int128)1 << j) < target) ++j;
  return j;
}

// Head counts are capped so that no workspace size can overflow size_t
// (the largest region, B Hkv (J+1) |pool| 8 bytes, stays below 2^60 with
// B <= 128, Hkv <= 1024, J + 1 <= 256 and n_max <= 2^31).
bool shape_ok(const csa_shape* s) {
  return s && s->B >= 1 && s->Hq >= 1 && s->Hkv >= 1 && s->Hq <= kMaxHeads && s->Hkv <= kMaxHeads &&
         s->Hq % s->Hkv == 0 && s->n_max >= 1 && s->n_max <= (int64_t)1 << 31 &&
         (s->dtype == CSA_BF16 || s->dtype == CSA_F32);
}
csa_status shape_supported(const csa_shape* s) {
  const int G = s->Hq / s->Hkv;
  if (s->d != 64 && s->d != 128) return CSA_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return CSA_ERR_UNSUPPORTED;
  if (s->B > kMaxB) return CSA_ERR_UNSUPPORTED;
  return CSA_OK;
}
bool params_ok(const csa_params* p) {
  return p && p->eps > 0.f && std::isfinite(p->eps) && p->delta > 0.f && p->delta < 1.f && p->r >= 1 &&
         p->r <= 4 && p->measure >= 0 && p->measure <= 3 && p->J_override >= -1 && p->J_override <= kMaxJ &&
         p->sub_batches >= 0 && p->sub_batches <= kMaxSub && (p->perturb == 0 || p->perturb == 1) &&
         (p->qcode == 0 || p->qcode == 1) && p->refine8 >= 0 && p->refine8 <= 2 && (p->dots == 0 || p->dots == 1);
}

// z with P(|N(0,1)| > z) = delta, i.e. erfc(z / sqrt 2) = delta: bisection
// on the decreasing function erfc (double precision, 200 halvings).
float normal_quantile_two_sided(double delta) {
  // the last delta's quantile is kept: the bisection costs ~10 us of host
  // time, and a decode loop asks for the same delta at every step
  static std::mutex mu;
  static double last_delta = -1.0;
  static float last_z = 0.f;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (delta == last_delta) return last_z;
  }
  double lo = 0.0, hi = 40.0;
  for (int i = 0; i < 200; ++i) {
    const double mid = 0.5 * (lo + hi);
    if (std::erfc(mid / std::sqrt(2.0)) > delta) lo = mid; else hi = mid;
  }
  const float z = (float)(0.5 * (lo + hi));
  std::lock_guard<std::mutex> lock(mu);
  last_delta = delta;
  last_z = z;
  return z;
}

struct Layout {
  int J1;
  int64_t pcap, nblk_max;
  size_t status, cmax, jr_hist, ncand, pre_hist, acc, bcnt, bcons, ccnt, xcnt, nfall, rq, front, jrd, ninset,
      zero_end;
  size_t jkey, jref, seqd, winstats, vmaxp, state, plan_start, plan_end, plan_off, ubar, hw, tmax, s32, win, t32, clist, xlist, cmap,
      buckets, dpart, pref, total;
  int64_t nchunk_cap;
};

bool make_layout(const csa_shape* s, const csa_params* p, Layout& L) {
  const int64_t B = s->B, Hq = s->Hq, Hkv = s->Hkv, D = s->d, G = Hq / Hkv;
  L.pcap = s->n_max > kWindow ? s->n_max - kWindow : 1;
  L.nblk_max = (s->n_max + kBlock - 1) / kBlock;
  const int Jmax = p->J_override >= 0 ? p->J_override : grid_J(L.pcap, p->r);
  if (Jmax > kMaxJ) return false;
  L.J1 = Jmax + 1;
  const int64_t BH = B * Hq, BG = B * Hkv, ACC = 2 * D + 8;
  size_t o = 0;
  L.status = o; o += up(64);
  L.cmax = o; o += up((size_t)BH * 4 * 4);
  L.jr_hist = o; o += up((size_t)BH * (L.J1 + 1) * 4);
  L.ncand = o; o += up((size_t)BH * 4);
  L.pre_hist = o; o += up((size_t)BH * L.J1 * 4 * 4);
  L.acc = o; o += up((size_t)BH * L.J1 * ACC * 4);
  L.bcnt = o; o += up((size_t)3 * BG * L.J1 * 4);
  L.bcons = o; o += up((size_t)BG * L.J1 * 4);
  L.ccnt = o; o += up((size_t)BG * 4);
  L.xcnt = o; o += up((size_t)BG * 4);
  L.nfall = o; o += up(4);
  L.rq = o; o += up(((size_t)BG * 6 + 6) * 4);
  L.front = o; o += up((size_t)4 * BG * 4);
  L.jrd = o; o += up(p->refine8 ? (size_t)BH * (L.J1 + 1) * 4 : 0);
  L.ninset = o; o += up(p->refine8 ? (size_t)BH * 4 : 0);
  L.zero_end = o;
  L.seqd = o; o += up(sizeof(SeqArgs) + sizeof(ReqPtrs));
  L.jkey = o; o += up(p->refine8 ? (size_t)BG * L.pcap * 2 : 0);
  L.jref = o; o += up(p->refine8 ? (size_t)BG * L.pcap * G * 2 : 0);
  L.winstats = o; o += up((size_t)BH * (D + 4) * 4);
  L.vmaxp = o; o += up((size_t)BG * 4);
  L.state = o; o += up((size_t)BH * 4 * 4);
  L.plan_start = o; o += up((size_t)BG * L.J1 * 4);
  L.plan_end = o; o += up((size_t)BG * L.J1 * 4);
  L.plan_off = o; o += up(((size_t)BG * L.J1 + 1) * 4);
  L.ubar = o; o += up((size_t)BG * s->n_max * G * 4);
  L.hw = o; o += up((size_t)BG * L.nblk_max * G * 4);
  L.tmax = o; o += up((size_t)BG * ((s->n_max + kTile - 1) / kTile) * G * 4);
  L.s32 = o; o += up((size_t)BG * L.pcap * G * 4);
  L.win = o; o += up((size_t)BG * kWindow * G * 4);
  L.t32 = o; o += up((size_t)BG * L.pcap * (p->perturb ? G : 1) * 4);
  L.clist = o; o += up((size_t)BG * L.pcap * 8);
  L.xlist = o; o += up((size_t)BG * s->n_max * 8);
  L.nchunk_cap = (int64_t)BG * L.J1 + (int64_t)BG * L.pcap * 2 * G / 1024 + 16;
  L.cmap = o; o += up((size_t)L.nchunk_cap * 4);
  L.buckets = o; o += up((size_t)BG * L.J1 * L.pcap * 8);
  L.dpart = o; o += up((size_t)dense_nsplit(s->n_max) * BH * (D + 2) * 4);
  L.pref = o; o += up((size_t)BH * ACC * 4);
  L.total = o;
  return true;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = v > 0 ? v : 148;
  }
  return cached[dev];
}

csa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA; }

// ----------------------------------------------------------- phase timing
constexpr int kProfSteps = 64;
constexpr int kProfEv = 2 * CSA_NPHASE + 8;   // boundaries per step (rounds repeat phases)
struct Profiler {
  bool on = false;
  bool made = false;
  cudaEvent_t ev[kProfSteps][kProfEv];
  int phase[kProfSteps][kProfEv];
  int nev[kProfSteps];
  int head = 0, count = 0, cur = -1;
  long long launches = 0;
};
Profiler g_prof;

void prof_step_begin(cudaStream_t st) {
  if (!g_prof.on) return;
  if (!g_prof.made) {
    for (int i = 0; i < kProfSteps; ++i)
      for (int j = 0; j < kProfEv; ++j) cudaEventCreate(&g_prof.ev[i][j]);
    g_prof.made = true;
  }
  g_prof.cur = (g_prof.head + g_prof.count) % kProfSteps;
  if (g_prof.count == kProfSteps) g_prof.head = (g_prof.head + 1) % kProfSteps;
  else ++g_prof.count;
  g_prof.nev[g_prof.cur] = 0;
  cudaEventRecord(g_prof.ev[g_prof.cur][0], st);
  g_prof.nev[g_prof.cur] = 1;
}
// mark the end of `phase` (the interval since the previous mark)
void prof_mark(int phase, cudaStream_t st) {
  if (!g_prof.on || g_prof.cur < 0) return;
  int k = g_prof.nev[g_prof.cur];
  if (k >= kProfEv) return;
  g_prof.phase[g_prof.cur][k] = phase;
  cudaEventRecord(g_prof.ev[g_prof.cur][k], st);
  g_prof.nev[g_prof.cur] = k + 1;
}
void count_launches(int k) { g_prof.launches += k; }

// ------------------------------------------------------------ sub-batches
//
// A batch of B >= 2 sequences runs by default as two sub-batches of
// consecutive sequences on library-owned streams: the step is a chain of
// ~20 dependent launches, several of them latency-bound, and independent
// chains fill the GPU better than one (128K x 4, chains enqueued stage by
// stage: one chain 814 us, two 686, four 694; each chain also costs ~50 us
// of host time to enqueue).  Each sub-batch has its
// own workspace region (stride `stride`); they share sub-batch 0's status
// word.

struct SubPlan {
  int nsub, Bc;
  size_t stride, total;
};

bool sub_plan(const csa_shape* s, const csa_params* p, SubPlan& sp) {
  Layout whole;
  if (!make_layout(s, p, whole)) return false;
  sp.nsub = p->sub_batches == 0 ? std::min(s->B, 2) : std::min(p->sub_batches, s->B);
  if (sp.nsub <= 1) {
    sp.nsub = 1; sp.Bc = s->B; sp.stride = whole.total; sp.total = whole.total;
    return true;
  }
  sp.Bc = (s->B + sp.nsub - 1) / sp.nsub;
  sp.nsub = (s->B + sp.Bc - 1) / sp.Bc;   // sub-batches that hold a sequence
  csa_shape sc = *s;
  sc.B = sp.Bc;
  Layout part;
  if (!make_layout(&sc, p, part)) return false;
  sp.stride = up(part.total);
  // room for the unsplit layout too (phase timing runs unsplit)
  sp.total = std::max(sp.stride * sp.nsub, whole.total);
  return true;
}

struct SubStreams {
  cudaStream_t st[kMaxSub];
  cudaEvent_t fork, join[kMaxSub];
  unsigned long long ctx;   // context the streams belong to
};
struct SubState {
  std::mutex mu;
  SubStreams* per_dev[64] = {nullptr};
};
SubState g_sub;

// the calling thread's device's streams and events, made on first use
// (callers hold g_sub.mu)
SubStreams* sub_streams() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  // the streams are keyed on the current context: after a device reset
  // they belong to a context that no longer exists, and are made again (the
  // old handles are dead).  (A caller of the step has device memory, so a
  // context is current; if none is, 0 stands for "made before any".)
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) ctx = 0;
  if (g_sub.per_dev[dev] && g_sub.per_dev[dev]->ctx != ctx) g_sub.per_dev[dev] = nullptr;
  if (!g_sub.per_dev[dev]) {
    SubStreams* ss = new SubStreams{};
    ss->ctx = ctx;
    bool ok = cudaEventCreateWithFlags(&ss->fork, cudaEventDisableTiming) == cudaSuccess;
    int made = 0;
    for (int c = 0; c < kMaxSub && ok; ++c) {
      ok = cudaStreamCreateWithFlags(&ss->st[c], cudaStreamNonBlocking) == cudaSuccess;
      if (ok && cudaEventCreateWithFlags(&ss->join[c], cudaEventDisableTiming) != cudaSuccess) {
        cudaStreamDestroy(ss->st[c]);
        ok = false;
      }
      if (ok) ++made;
    }
    if (!ok) {
      // release what was made; a later call tries again
      for (int c = 0; c < made; ++c) {
        cudaStreamDestroy(ss->st[c]);
        cudaEventDestroy(ss->join[c]);
      }
      if (ss->fork) cudaEventDestroy(ss->fork);
      delete ss;
      return nullptr;
    }
    g_sub.per_dev[dev] = ss;
  }
  return g_sub.per_dev[dev];
}

// Where a step's per-sequence lengths and seeds come from: host arrays
// (copied into the launch arguments) or device arrays (read by a first
// kernel into the workspace; grids are then sized from the capacity n_max).
struct SeqSource {
  const int64_t* len;
  const uint64_t* seed;
  bool dev;
  bool requant;            // device lengths: re-quantise the block of token len - 1
  uint8_t* K4w;
  float* boundsw;
  float* vmaxw;
  float* vnorm2w;
  const uint8_t* K8;       // 8-bit codes and steps (refinement tier), or null
  const float* delta8;
};

// One (sub-)batch on one stream, as a chain of launch stages.  `status` is
// the device status word (shared by the sub-batches of a split call);
// `clear` zeroes the per-step counters (a split call clears sub-batch 0's,
// which hold the status word, before it forks).  A split call enqueues the
// chains stage by stage (stage k of every chain, then stage k + 1), so every
// chain starts on the device while the host is still enqueueing the rest.
struct Chain {
  csa_shape shape;
  const csa_params* params;
  SeqSource src;
  Layout L;
  SeqArgs seq;
  ScanArgs sa;
  SparseArgs a;
  DenseArgs da;
  int64_t nlive, plive;
  int G;
  bool bf16, clear, stats;
  bool tm_ok;             // tm_codes holds a tensor map of the code rows
  CUtensorMap tm_codes;
  char* ws;
  unsigned* status;
  cudaStream_t st;
};
constexpr int kChainStages = 10;
#ifndef CSA_SCAN_TMA
#define CSA_SCAN_TMA 1
#endif
constexpr bool kScanTma = CSA_SCAN_TMA != 0;   // bulk tensor staging of the scan's code tiles

csa_status chain_prepare(Chain& c, const csa_shape* shape, const csa_params* params, const void* q,
                         const void* K, const void* V, const uint8_t* K4, const float* bounds, const float* vmax,
                         const float* vnorm2, const SeqSource& src, float* o, float* beta, int32_t* level,
                         int32_t* keys_read, csa_head_stats* stats, char* ws, unsigned* status, bool clear,
                         cudaStream_t st) {
  c.shape = *shape;
  c.params = params;
  c.src = src;
  c.ws = ws;
  c.status = status;
  c.clear = clear;
  c.st = st;
  c.stats = stats != nullptr;
  Layout& L = c.L;
  if (!make_layout(shape, params, L)) return CSA_ERR_INVALID_ARG;
  c.G = shape->Hq / shape->Hkv;
  c.bf16 = shape->dtype == CSA_BF16;
  std::memset(&c.seq, 0, sizeof(c.seq));
  int64_t nlive = 0;
  const SeqArgs* seqd = nullptr;
  if (!src.dev) {
    for (int b = 0; b < shape->B; ++b) {
      const int64_t n = src.len[b];
      if (n < 1 || n > shape->n_max) return CSA_ERR_INVALID_ARG;
      c.seq.n[b] = n;
      c.seq.seed[b] = src.seed[b];
      const int64_t P = n > kWindow ? n - kWindow : 0;
      c.seq.J[b] = params->J_override >= 0 ? params->J_override : grid_J(P, params->r);
      if (n > nlive) nlive = n;
    }
  } else {
    nlive = shape->n_max;
    seqd = (const SeqArgs*)(ws + L.seqd);
  }
  c.nlive = nlive;
  c.plive = nlive > kWindow ? nlive - kWindow : 0;
  const float rs = (float)(1.0 / std::sqrt((double)shape->d));

  ScanArgs& sa = c.sa;
  sa = {};
  sa.q = q; sa.K4 = K4; sa.bounds = bounds; sa.ubar = (float*)(ws + L.ubar);
  sa.hw = (float*)(ws + L.hw);
  sa.tmax = (float*)(ws + L.tmax);
  sa.cmax = (unsigned*)(ws + L.cmax); sa.status = status;
  sa.Hq = shape->Hq; sa.Hkv = shape->Hkv; sa.n_max = shape->n_max; sa.nblk_max = L.nblk_max; sa.rs = rs;
  sa.two_digit = params->qcode == 1;
  sa.seqd = seqd;
  sa.requant = src.dev && src.requant;
  sa.dp4a = params->dots == 1;
  // the plain d = 128 scan stages its code tile with one bulk tensor copy
  // (64-byte rows, 256-row boxes; the row index must fit in int32)
  {
    const uint64_t crows = (uint64_t)shape->B * shape->Hkv * L.nblk_max * kBlock;
    c.tm_ok = kScanTma && shape->d == 128 && !sa.requant && !sa.two_digit && !sa.dp4a && crows < (1ull << 31) &&
              make_tmap_2d_u8_sw64(&c.tm_codes, K4, 64, crows, 64, 64, kTile);
  }

  SparseArgs& a = c.a;
  a = {};
  a.q = q; a.K = K; a.V = V; a.vmax = vmax; a.vnorm2 = vnorm2; a.ubar = (const float*)(ws + L.ubar);
  a.s32 = (float*)(ws + L.s32); a.win = (float*)(ws + L.win); a.cmax = (unsigned*)(ws + L.cmax);
  a.jr_hist = (unsigned*)(ws + L.jr_hist); a.ncand = (unsigned*)(ws + L.ncand);
  a.pre_hist = (float*)(ws + L.pre_hist); a.acc = (float*)(ws + L.acc); a.winstats = (float*)(ws + L.winstats);
  a.vmaxp = (float*)(ws + L.vmaxp); a.state = (int*)(ws + L.state); a.bcnt = (unsigned*)(ws + L.bcnt);
  a.bcons = (unsigned*)(ws + L.bcons); a.buckets = (uint2*)(ws + L.buckets);
  a.t32 = (float*)(ws + L.t32); a.clist = (uint2*)(ws + L.clist); a.ccnt = (unsigned*)(ws + L.ccnt);
  a.nfall = (unsigned*)(ws + L.nfall);
  a.rq = (unsigned*)(ws + L.rq);
  a.pref = (float*)(ws + L.pref);
  a.hw = (const float*)(ws + L.hw); a.tmax = (const float*)(ws + L.tmax); a.front = (int*)(ws + L.front);
  a.xlist = (uint2*)(ws + L.xlist); a.xcnt = (unsigned*)(ws + L.xcnt);
  a.chunk_map = (unsigned*)(ws + L.cmap); a.nchunk_cap = L.nchunk_cap;
  a.plan_start = (unsigned*)(ws + L.plan_start); a.plan_end = (unsigned*)(ws + L.plan_end);
  a.plan_off = (unsigned*)(ws + L.plan_off); a.status = status;
  a.o = o; a.beta = beta; a.level = level; a.keys_read = keys_read; a.stats = stats;
  a.B = shape->B; a.Hq = shape->Hq; a.Hkv = shape->Hkv; a.n_max = shape->n_max; a.nblk_max = L.nblk_max;
  a.pcap = L.pcap; a.J1 = L.J1; a.r = params->r; a.eps = params->eps; a.delta = params->delta;
  a.measure = params->measure; a.rs = rs; a.per_head = params->perturb;
  a.zclt = normal_quantile_two_sided((double)params->delta);
  a.seqd = seqd;
  a.refine8 = params->refine8;
  if (params->refine8) {
    a.K8 = src.K8; a.delta8 = src.delta8; a.bounds = bounds;
    a.jkey = (uint16_t*)(ws + L.jkey); a.jrd = (int*)(ws + L.jrd); a.ninset = (unsigned*)(ws + L.ninset);
    a.jref = (uint16_t*)(ws + L.jref);
  }

  // exact attention for heads with no certified level and sequences without a pool
  DenseArgs& da = c.da;
  da = {};
  da.q = q; da.K = K; da.V = V; da.part = (float*)(ws + L.dpart); da.o = o; da.state = a.state;
  da.nfall = a.nfall;
  da.status = status;
  da.seqd = seqd;
  da.B = shape->B; da.Hq = shape->Hq; da.Hkv = shape->Hkv; da.n_max = shape->n_max;
  da.nsplit = dense_nsplit(shape->n_max); da.rs = rs;
  return CSA_OK;
}

csa_status chain_stage(Chain& c, int stage, int nsm) {
  const csa_params* params = c.params;
  cudaStream_t st = c.st;
  const int d = c.shape.d, G = c.G;
  switch (stage) {
    case 0:
      prof_step_begin(st);
      if (c.clear && cudaMemsetAsync(c.ws, 0, c.L.zero_end, st) != cudaSuccess) return CSA_ERR_CUDA;
      if (c.src.dev) {
        const ReqPtrs req = {c.a.K, c.a.V, c.src.K4w, c.src.boundsw, c.src.vmaxw, c.src.vnorm2w};
        if (launch_seq_prep(c.src.len, c.src.seed, c.shape.B, c.shape.n_max, params->r, params->J_override,
                            (SeqArgs*)(c.ws + c.L.seqd), req, c.status, st) != cudaSuccess)
          return CSA_ERR_CUDA;
        count_launches(1);
      }
      prof_mark(0, st);
      return CSA_OK;
    case 1:
      if (launch_scan(c.sa, c.seq, c.shape.B, d, G, c.bf16, c.nlive, c.tm_ok ? &c.tm_codes : nullptr, st) !=
          cudaSuccess)
        return CSA_ERR_CUDA;
      count_launches(1);
      prof_mark(1, st);
      return CSA_OK;
    case 2:
      if (c.plive > 0) {
        if (launch_cstar(c.a, c.seq, d, G, c.bf16, c.nlive, nsm, st) != cudaSuccess) return CSA_ERR_CUDA;
        count_launches(2);
        prof_mark(2, st);
      }
      return CSA_OK;
    case 3:
      if (c.plive > 0) {
        if (launch_candidates(c.a, c.seq, G, c.plive, nsm, st) != cudaSuccess) return CSA_ERR_CUDA;
        count_launches(1);
        prof_mark(3, st);
      }
      return CSA_OK;
    case 4:
      if (launch_predict(c.a, c.seq, d, G, c.bf16, st) != cudaSuccess) return CSA_ERR_CUDA;
      count_launches(1);
      prof_mark(5, st);
      return CSA_OK;
    case 5:
    case 6:
    case 7: {
      const int round = stage - 5;
      if (launch_round(c.a, c.seq, d, G, c.bf16, c.plive > 0 ? c.plive : 1, round, nsm, st,
                       g_prof.on ? prof_mark : nullptr) != cudaSuccess)
        return CSA_ERR_CUDA;
      count_launches(4);
      return CSA_OK;
    }
    case 8:
      if (launch_dense(c.da, c.seq, d, G, c.bf16, c.nlive, st) != cudaSuccess) return CSA_ERR_CUDA;
      count_launches(2);
      prof_mark(10, st);
      return CSA_OK;
    case 9:
      if (c.stats && c.plive > 0) {
        if (launch_near(c.a, c.seq, G, c.plive, st) != cudaSuccess) return CSA_ERR_CUDA;
        count_launches(1);
        prof_mark(11, st);
      }
      return CSA_OK;
    default:
      return CSA_OK;
  }
}

}  // namespace

void add_launches(int k) { count_launches(k); }

namespace {
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, CUtensorMapSwizzle sw, const void* base, uint64_t inner,
                  uint64_t rows, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows) {
  typedef CUresult (*Encode)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                             CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static std::once_flag once;
  static Encode encode = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = (Encode)f;
  });
  if (!encode || !base || ((uintptr_t)base & 15u) || (pitch_bytes & 15u)) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                       uint32_t box_inner, uint32_t box_rows) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, base, inner, rows,
                      pitch_bytes, box_inner, box_rows);
}

bool make_tmap_2d_u8_sw64(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint64_t pitch_bytes,
                          uint32_t box_inner, uint32_t box_rows) {
  return make_tmap_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_64B, base, inner, rows, pitch_bytes,
                      box_inner, box_rows);
}

bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrent)(CUcontext*);
  typedef CUresult (*GetId)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = (GetCurrent)f;
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = (GetId)f;
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace csa

using namespace csa;

extern "C" {

const char* csa_status_string(csa_status s) {
  switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID_ARG: return "invalid argument";
    case CSA_ERR_UNSUPPORTED: return "unsupported shape (d must be 64 or 128, G in {1,2,4,8}, B <= 128)";
    case CSA_ERR_CUDA: return "CUDA error";
    case CSA_ERR_NONFINITE: return "non-finite value in q, K or the statistics";
    case CSA_ERR_TIMEOUT: return "device wait timed out";
    case CSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

size_t csa_workspace_size(const csa_shape* shape, const csa_params* params) {
  if (!shape_ok(shape) || !params_ok(params) || shape_supported(shape) != CSA_OK) return 0;
  SubPlan sp;
  if (!sub_plan(shape, params, sp)) return 0;
  return sp.total;
}

// dense workspace: the status word (256 bytes), then the split-K partials
size_t csa_dense_workspace_size(const csa_shape* shape) {
  if (!shape_ok(shape) || shape_supported(shape) != CSA_OK) return 0;
  return kAlign + up((size_t)dense_nsplit(shape->n_max) * shape->B * shape->Hq * (shape->d + 2) * 4);
}

csa_status csa_workspace_layout(const csa_shape* shape, const csa_params* params, csa_workspace_map* out) {
  if (!out || !shape_ok(shape) || !params_ok(params)) return CSA_ERR_INVALID_ARG;
  csa_status su = shape_supported(shape);
  if (su != CSA_OK) return su;
  SubPlan sp;
  if (!sub_plan(shape, params, sp)) return CSA_ERR_INVALID_ARG;
  csa_shape s0 = *shape;
  s0.B = sp.Bc;
  Layout L;
  if (!make_layout(&s0, params, L)) return CSA_ERR_INVALID_ARG;
  out->ubar = L.ubar;
  out->cmax = L.cmax;
  out->s32 = L.s32;
  out->jr_hist = L.jr_hist;
  out->bcnt = L.bcons;   // cumulative over the step's rounds
  out->total = sp.total;
  out->J1 = L.J1;
  out->sub_batches = sp.nsub;
  out->sub_stride = sp.stride;
  out->sub_B = sp.Bc;
  return CSA_OK;
}

csa_status csa_quantize_keys(const csa_shape* shape, const void* K, const void* V, const int64_t* len,
                             int64_t from_token, uint8_t* K4, float* bounds, float* vmax, float* vnorm2,
                             void* stream) {
  if (!shape_ok(shape) || !K || !V || !len || !K4 || !bounds || !vmax || !vnorm2 || from_token < 0)
    return CSA_ERR_INVALID_ARG;
  csa_status su = shape_supported(shape);
  if (su != CSA_OK) return su;
  SeqArgs seq;
  std::memset(&seq, 0, sizeof(seq));
  int64_t nblocks = 0;
  const int64_t blk_from = from_token / kBlock;
  for (int b = 0; b < shape->B; ++b) {
    if (len[b] < 0 || len[b] > shape->n_max) return CSA_ERR_INVALID_ARG;
    seq.n[b] = len[b];
    const int64_t nb = (len[b] + kBlock - 1) / kBlock - blk_from;
    if (nb > nblocks) nblocks = nb;
  }
  QuantArgs a = {};
  a.K = K; a.V = V; a.K4 = K4; a.bounds = bounds; a.vmax = vmax; a.vnorm2 = vnorm2; a.Hkv = shape->Hkv;
  a.n_max = shape->n_max; a.nblk_max = (shape->n_max + kBlock - 1) / kBlock; a.blk_from = blk_from;
  if (nblocks > 0) count_launches(1);
  return cuda_status(launch_quant(a, seq, shape->B, shape->d, shape->dtype == CSA_BF16, nblocks,
                                  (cudaStream_t)stream));
}

csa_status csa_quantize_keys8(const csa_shape* shape, const void* K, const int64_t* len, int64_t from_token,
                              uint8_t* K8, float* delta8, void* stream) {
  if (!shape_ok(shape) || !K || !len || !K8 || !delta8 || from_token < 0) return CSA_ERR_INVALID_ARG;
  csa_status su = shape_supported(shape);
  if (su != CSA_OK) return su;
  SeqArgs seq;
  std::memset(&seq, 0, sizeof(seq));
  int64_t nblocks = 0;
  const int64_t blk_from = from_token / kBlock;
  for (int b = 0; b < shape->B; ++b) {
    if (len[b] < 0 || len[b] > shape->n_max) return CSA_ERR_INVALID_ARG;
    seq.n[b] = len[b];
    const int64_t nb = (len[b] + kBlock - 1) / kBlock - blk_from;
    if (nb > nblocks) nblocks = nb;
  }
  QuantArgs a = {};
  a.K = K; a.K8 = K8; a.delta8 = delta8; a.Hkv = shape->Hkv;
  a.n_max = shape->n_max; a.nblk_max = (shape->n_max + kBlock - 1) / kBlock; a.blk_from = blk_from;
  if (nblocks > 0) count_launches(1);
  return cuda_status(launch_quant8(a, seq, shape->B, shape->d, shape->dtype == CSA_BF16, nblocks,
                                   (cudaStream_t)stream));
}

csa_status csa_dense_decode(const csa_shape* shape, const void* q, const void* K, const void* V,
                            const int64_t* len, float* o, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!shape_ok(shape) || !q || !K || !V || !len || !o) return CSA_ERR_INVALID_ARG;
  csa_status su = shape_supported(shape);
  if (su != CSA_OK) return su;
  const size_t need = csa_dense_workspace_size(shape);
  if (!workspace || workspace_bytes < need || ((uintptr_t)workspace % kAlign)) return CSA_ERR_WORKSPACE;
  SeqArgs seq;
  std::memset(&seq, 0, sizeof(seq));
  int64_t nlive = 0;
  for (int b = 0; b < shape->B; ++b) {
    if (len[b] < 1 || len[b] > shape->n_max) return CSA_ERR_INVALID_ARG;
    seq.n[b] = len[b];
    if (len[b] > nlive) nlive = len[b];
  }
  if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), (cudaStream_t)stream) != cudaSuccess) return CSA_ERR_CUDA;
  DenseArgs a = {};
  a.q = q; a.K = K; a.V = V; a.part = (float*)((char*)workspace + kAlign); a.o = o; a.state = nullptr;
  a.nfall = nullptr; a.status = (unsigned*)workspace;
  a.B = shape->B; a.Hq = shape->Hq; a.Hkv = shape->Hkv; a.n_max = shape->n_max;
  a.nsplit = dense_nsplit(shape->n_max); a.rs = (float)(1.0 / std::sqrt((double)shape->d));
  count_launches(2);
  return cuda_status(launch_dense(a, seq, shape->d, shape->Hq / shape->Hkv, shape->dtype == CSA_BF16, nlive,
                                  (cudaStream_t)stream));
}

}  // extern "C"

namespace csa {
namespace {

// The step for host or device lengths: checks, then one chain or the
// sub-batch fork.
csa_status decode_step_impl(const csa_shape* shape, const csa_params* params, const void* q, const void* K,
                            const void* V, const uint8_t* K4, const float* bounds, const float* vmax,
                            const float* vnorm2, const SeqSource& src, float* o, float* beta, int32_t* level,
                            int32_t* keys_read, csa_head_stats* stats, void* workspace, size_t workspace_bytes,
                            void* stream) {
  if (!shape_ok(shape) || !params_ok(params) || !q || !K || !V || !K4 || !bounds || !vmax || !vnorm2 ||
      !src.len || !src.seed || !o || !beta || !level || !keys_read)
    return CSA_ERR_INVALID_ARG;
  if (params->refine8 && (!src.K8 || !src.delta8)) return CSA_ERR_INVALID_ARG;
  csa_status su = shape_supported(shape);
  if (su != CSA_OK) return su;
  if (params->refine8 && shape->dtype != CSA_BF16) return CSA_ERR_UNSUPPORTED;
  SubPlan sp;
  if (!sub_plan(shape, params, sp)) return CSA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < sp.total || ((uintptr_t)workspace % kAlign)) return CSA_ERR_WORKSPACE;
  if (!src.dev)
    for (int b = 0; b < shape->B; ++b)
      if (src.len[b] < 1 || src.len[b] > shape->n_max) return CSA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  char* ws = (char*)workspace;
  unsigned* status = (unsigned*)ws;   // offset 0 of (sub-batch 0's) layout
  const int nsm = sm_count();
  if (sp.nsub == 1 || g_prof.on) {
    // one stream (phase timing runs unsplit so its events bracket whole phases)
    Chain c;
    csa_status r = chain_prepare(c, shape, params, q, K, V, K4, bounds, vmax, vnorm2, src, o, beta, level,
                                 keys_read, stats, ws, status, true, st);
    for (int k = 0; r == CSA_OK && k < kChainStages; ++k) r = chain_stage(c, k, nsm);
    return r;
  }
  // sub-batches of consecutive sequences on the library's streams: fork
  // after clearing sub-batch 0's counters (they hold the status word), join
  // back onto the caller's stream
  std::lock_guard<std::mutex> lock(g_sub.mu);
  SubStreams* ss = sub_streams();
  if (!ss) return CSA_ERR_CUDA;
  {
    csa_shape s0 = *shape;
    s0.B = sp.Bc;
    Layout L0;
    if (!make_layout(&s0, params, L0)) return CSA_ERR_INVALID_ARG;
    if (cudaMemsetAsync(ws, 0, L0.zero_end, st) != cudaSuccess) return CSA_ERR_CUDA;
  }
  if (cudaEventRecord(ss->fork, st) != cudaSuccess) return CSA_ERR_CUDA;
  const size_t esz = shape->dtype == CSA_BF16 ? 2 : 4;
  const int64_t nblk = (shape->n_max + kBlock - 1) / kBlock;
  const int64_t Hq = shape->Hq, Hkv = shape->Hkv, D = shape->d, N = shape->n_max;
  Chain chains[kMaxSub];
  int nch = 0;
  for (int c = 0; c < sp.nsub; ++c) {
    const int64_t b0 = (int64_t)c * sp.Bc;
    if (b0 >= shape->B) break;
    csa_shape sc = *shape;
    sc.B = (int)std::min<int64_t>(sp.Bc, shape->B - b0);
    cudaStream_t cs = ss->st[c];
    if (cudaStreamWaitEvent(cs, ss->fork, 0) != cudaSuccess) return CSA_ERR_CUDA;
    SeqSource sc_src = src;
    sc_src.len = src.len + b0;
    sc_src.seed = src.seed + b0;
    if (src.requant) {
      sc_src.K4w = src.K4w + b0 * Hkv * nblk * kBlock * (D / 2);
      sc_src.boundsw = src.boundsw + b0 * Hkv * nblk * 2 * D;
      sc_src.vmaxw = src.vmaxw + b0 * Hkv * nblk;
      sc_src.vnorm2w = src.vnorm2w + b0 * Hkv * N;
    }
    if (src.K8) {
      sc_src.K8 = src.K8 + b0 * Hkv * nblk * kBlock * D;
      sc_src.delta8 = src.delta8 + b0 * Hkv * nblk * D;
    }
    csa_status r = chain_prepare(
        chains[nch], &sc, params, (const char*)q + b0 * Hq * D * esz, (const char*)K + b0 * Hkv * N * D * esz,
        (const char*)V + b0 * Hkv * N * D * esz, K4 + b0 * Hkv * nblk * kBlock * (D / 2),
        bounds + b0 * Hkv * nblk * 2 * D, vmax + b0 * Hkv * nblk, vnorm2 + b0 * Hkv * N, sc_src,
        o + b0 * Hq * D, beta + b0 * Hq, level + b0 * Hq, keys_read + b0 * Hq,
        stats ? stats + b0 * Hq : nullptr, ws + c * sp.stride, status, c > 0, cs);
    if (r != CSA_OK) return r;
    ++nch;
  }
  // stage k of every chain, then stage k + 1
  for (int k = 0; k < kChainStages; ++k)
    for (int c = 0; c < nch; ++c) {
      const csa_status r = chain_stage(chains[c], k, nsm);
      if (r != CSA_OK) return r;
    }
  for (int c = 0; c < nch; ++c) {
    if (cudaEventRecord(ss->join[c], ss->st[c]) != cudaSuccess) return CSA_ERR_CUDA;
    if (cudaStreamWaitEvent(st, ss->join[c], 0) != cudaSuccess) return CSA_ERR_CUDA;
  }
  return CSA_OK;
}

}  // namespace
}  // namespace csa

extern "C" {

csa_status csa_decode_step(const csa_shape* shape, const csa_params* params, const void* q, const void* K,
                           const void* V, const uint8_t* K4, const float* bounds, const float* vmax,
                           const float* vnorm2, const int64_t* len, const uint64_t* step_seed, float* o,
                           float* beta, int32_t* level, int32_t* keys_read, csa_head_stats* stats, void* workspace,
                           size_t workspace_bytes, void* stream) {
  SeqSource src = {len, step_seed, false, false, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  return decode_step_impl(shape, params, q, K, V, K4, bounds, vmax, vnorm2, src, o, beta, level, keys_read, stats,
                          workspace, workspace_bytes, stream);
}

csa_status csa_decode_step_refined(const csa_shape* shape, const csa_params* params, const void* q, const void* K,
                                   const void* V, const uint8_t* K4, const float* bounds, const float* vmax,
                                   const float* vnorm2, const uint8_t* K8, const float* delta8, const int64_t* len,
                                   const uint64_t* step_seed, float* o, float* beta, int32_t* level,
                                   int32_t* keys_read, csa_head_stats* stats, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  if (!K8 || !delta8) return CSA_ERR_INVALID_ARG;
  SeqSource src = {len, step_seed, false, false, nullptr, nullptr, nullptr, nullptr, K8, delta8};
  return decode_step_impl(shape, params, q, K, V, K4, bounds, vmax, vnorm2, src, o, beta, level, keys_read, stats,
                          workspace, workspace_bytes, stream);
}

csa_status csa_decode_step_device(const csa_shape* shape, const csa_params* params, const void* q, const void* K,
                                  const void* V, uint8_t* K4, float* bounds, float* vmax, float* vnorm2,
                                  const int64_t* len, const uint64_t* step_seed, int requantize_last, float* o,
                                  float* beta, int32_t* level, int32_t* keys_read, csa_head_stats* stats,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (requantize_last != 0 && requantize_last != 1) return CSA_ERR_INVALID_ARG;
  if (params && params->refine8) return CSA_ERR_INVALID_ARG;   // (the refinement takes host lengths)
  SeqSource src = {len, step_seed, true, requantize_last == 1, K4, bounds, vmax, vnorm2, nullptr, nullptr};
  return decode_step_impl(shape, params, q, K, V, K4, bounds, vmax, vnorm2, src, o, beta, level, keys_read, stats,
                          workspace, workspace_bytes, stream);
}

csa_status csa_profile_enable(int on) {
  g_prof.on = on != 0;
  return CSA_OK;
}

csa_status csa_profile_read(csa_phase_times* out) {
  if (!out) return CSA_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  for (int c = 0; c < g_prof.count; ++c) {
    const int i = (g_prof.head + c) % kProfSteps;
    if (g_prof.nev[i] < 2) continue;
    if (cudaEventSynchronize(g_prof.ev[i][g_prof.nev[i] - 1]) != cudaSuccess) return CSA_ERR_CUDA;
    for (int k = 1; k < g_prof.nev[i]; ++k) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, g_prof.ev[i][k - 1], g_prof.ev[i][k]) != cudaSuccess) return CSA_ERR_CUDA;
      out->ms[g_prof.phase[i][k]] += ms;
    }
    out->steps += 1;
  }
  out->launches = g_prof.launches;
  g_prof.head = 0;
  g_prof.count = 0;
  g_prof.cur = -1;
  g_prof.launches = 0;
  return CSA_OK;
}

csa_status csa_check(void* workspace, void* stream) {
  if (!workspace) return CSA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaStreamSynchronize(st) != cudaSuccess) return CSA_ERR_CUDA;
  unsigned w = 0;
  if (cudaMemcpy(&w, workspace, sizeof(w), cudaMemcpyDeviceToHost) != cudaSuccess) return CSA_ERR_CUDA;
  if (w & 1u) return CSA_ERR_NONFINITE;
  if (w & 2u) return CSA_ERR_WORKSPACE;
  if (w & 4u) return CSA_ERR_TIMEOUT;
  if (w & 8u) return CSA_ERR_INVALID_ARG;
  return CSA_OK;
}

}  // extern "C"
