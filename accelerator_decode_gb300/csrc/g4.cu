// libg4: C ABI of the GB300 greedy decode step (see include/g4.h).
//
// One decode step, for n sequences (launch order; every kernel reads only what earlier
// launches on the stream wrote):
//   embed            x0 = E[t] sqrt(H); tok = T_ple[t] sqrt(P)
//   gemv pmp         pr = W_pmp x0
//   ple_combine      ple_l = (RMSNorm(pr_l H^-1/2) + tok_l) / sqrt 2
//   per layer l:
//     gemv qkv       prologue x = (x + RMSNorm(r_ple)) lambda_{l-1}; h = RMSNorm(x); y = W_qkv h
//     attention      q/k norm + RoPE, K/V write (owning layers), flash-decode over cache[src]
//     gemv o         r_attn = W_o o
//     gemv gate/up   prologue x += RMSNorm(r_attn); m = RMSNorm(x); act = gelu(W_g m) * (W_u m)
//     gemv down      r_mlp = W_d act
//     gemv ple_gate  prologue x += RMSNorm(r_mlp); g = gelu(W_pg x) * ple_l
//     gemv ple_proj  r_ple = W_pp g
//   gemv lm_head     prologue x = (x + RMSNorm(r_ple)) lambda; y = RMSNorm(x); logits = E y,
//                    block argmax + last-block reduction -> next ids
// "gemv" is the tiled GEMV for up to 4 rows and the tcgen05 GEMM (with an activation-prep
// kernel for the prologue) from 5 rows.  Decode steps are captured into a CUDA graph per
// (n, step mode, pointer set) and replayed; g4_set_step_mode(1) runs steps of 1-2 rows as one
// persistent launch instead (mega.cuh).  Prefill runs blocks of up to 64 prompt rows through
// the same step with the K/V rows written ahead of each attention (kv_first).
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "attn.cuh"
#include "attn_mqa.cuh"
#include "common.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"
#include "gemv_s.cuh"
#include "mega.cuh"
#include "misc.cuh"

using namespace g4;

namespace {

thread_local std::string g_last_cuda;

bool cuda_ok(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return true;
  char buf[512];
  snprintf(buf, sizeof buf, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  g_last_cuda = buf;
  return false;
}
#define CK(call)                                           \
  do {                                                     \
    if (!cuda_ok((call), #call)) return G4_ERR_CUDA;       \
  } while (0)

// Makes `dev` current for the guard's lifetime and gives the caller's current device back
// afterwards, so no entry point changes the calling thread's device.
struct DeviceGuard {
  int prev = -1, dev = -1;
  cudaError_t err = cudaSuccess;
  explicit DeviceGuard(int d) : dev(d) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) err = cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0 && prev != dev) cudaSetDevice(prev);
  }
};
#define DEVICE_GUARD(d)   \
  DeviceGuard dg_guard_(d); \
  CK(dg_guard_.err)

inline int cdiv(int a, int b) { return (a + b - 1) / b; }

struct Seg {
  const void* w;
  const void* s;
  int rows;
};

// A projection in the tiled layout with its launch plan.
struct Lin {
  int fmt = 0, N = 0, K = 0, n_rb = 0, S = 0, tiles = 0, R = 1;
  int n_valid = 0;  // outputs
  int sg_per_cta = 1, ksplit = 1;
  uint4* qw = nullptr;
  uint4* sc = nullptr;
  size_t bytes = 0;
};

struct Layer {
  int full = 0, d = 0, F = 0, own = 0, src = 0, kv = -1;
  Lin qkv, o, gu, down, pg, pp;
  const __nv_bfloat16 *in_norm, *post_attn_norm, *pre_ffw_norm, *post_ffw_norm, *post_ple_norm, *q_norm, *k_norm;
  float lambda = 1.f;
  float scale = 1.f;
  int attn_hpc = 1;
};

struct GraphKey {
  int n, mode;
  const void *slots, *tokens, *pos, *next, *logits, *trace;
  bool operator<(const GraphKey& o) const {
    return std::tie(n, mode, slots, tokens, pos, next, logits, trace) <
           std::tie(o.n, o.mode, o.slots, o.tokens, o.pos, o.next, o.logits, o.trace);
  }
};

}  // namespace

struct g4_handle {
  g4_config cfg{};
  int device = 0, sms = 0;
  std::vector<void*> allocs;
  size_t bytes = 0;
  // allocation-failure injection (tests): the fail_at-th device allocation of g4_create
  // reports out-of-memory without allocating (G4_FAIL_ALLOC_AT; 0 = off)
  int fail_at = 0, n_allocs = 0;
  int* probe_flag = nullptr;  // a flag nothing sets (g4_timeout_probe)
  std::vector<Layer> layers;
  Lin pmp, lm;
  const __nv_bfloat16 *embed = nullptr, *ple_table = nullptr, *g_ppn = nullptr, *g_final = nullptr;
  // int4 vocabulary tables (table_format G4_W4A16): borrowed words and scales; the lm_head
  // is then an int4 projection built from the embedding's
  bool t4 = false;
  const uint32_t *embed_q = nullptr, *ple_q = nullptr;
  const __nv_bfloat16 *embed_s = nullptr, *ple_s = nullptr;
  // KV cache per owning layer: rows of d values (bf16, or int8 codes with an fp32 scale per
  // row in ksc / vsc).  Static rows: slot * max_context + position.  Paged: a pool of n_pages
  // pages of 2^page_shift rows per layer, one page table for all layers (device copy
  // page_table [max_batch][max_pages], host mirror pt_host), free pages in free_pages.
  std::vector<void*> kc, vc;
  std::vector<float*> ksc, vsc;
  bool kv8 = false;
  int* page_table = nullptr;
  int page_shift = 0, max_pages = 0, n_pages = 0;
  std::vector<int> pt_host, slot_pages, free_pages;
  float *cos_t[2] = {nullptr, nullptr}, *sin_t[2] = {nullptr, nullptr};
  // activations
  float *x0 = nullptr, *xb[2] = {nullptr, nullptr}, *tok = nullptr, *pr = nullptr, *ple = nullptr;
  float *qkv = nullptr, *attn = nullptr, *r_attn = nullptr, *act = nullptr, *r_mlp = nullptr, *pg = nullptr,
        *r_ple = nullptr;
  // scratch
  float* gemv_part = nullptr;
  unsigned* gemv_cnt = nullptr;
  size_t gemv_part_floats = 0, gemv_cnt_n = 0;
  float* am_val = nullptr;
  int* am_idx = nullptr;
  size_t am_n = 0;
  uint8_t* xt = nullptr;  // tensor-core GEMM activation tiles
  size_t xt_bytes = 0;
  float* tc_part = nullptr;
  size_t tc_part_floats = 0;
  float *attn_ml = nullptr, *attn_o = nullptr;
  unsigned* attn_cnt = nullptr;
  size_t attn_ml_n = 0, attn_o_n = 0;
  int* err = nullptr;
  // prefill staging
  int* pf_buf = nullptr;
  // staged decode step (1-4 rows): row-group counters per staged launch of a step, and the
  // raw K-slice partial sums each projection hands to the next kernel ([kSgMaxParts][4][width])
  unsigned* sg_ctr = nullptr;
  float *sq_qkv = nullptr, *sq_rattn = nullptr, *sq_gu = nullptr, *sq_rmlp = nullptr, *sq_pg = nullptr,
        *sq_rple = nullptr, *sq_pr = nullptr;
  int sq_qkv_w = 0, sq_gu_w = 0;
  size_t pf_cap = 0;
  int* step_next = nullptr;
  float* step_logits = nullptr;
  // trace
  float* trace = nullptr;
  int trace_stride = 0;
  // persistent step (n <= 2)
  int rows = 0;    // activation rows the step buffers hold (>= max_batch)
  int l_tail = 0;  // layers [l_tail, num_layers) write no K/V
  bool mega_ok = false;  // the persistent step was planned for this model
  bool mega_on = false;  // g4_set_step_mode(1): n_seq <= 2 steps run it
  MegaPhase* mega_phases = nullptr;
  int mega_n = 0, mega_grid = 0;
  size_t mega_smem = 0;
  unsigned* mega_bar = nullptr;
  unsigned long long* mega_stamps = nullptr;
  std::vector<std::string> mega_names;  // phase names (profiling)
  float *mega_am_val = nullptr;
  int* mega_am_idx = nullptr;
  // graphs
  std::map<GraphKey, cudaGraphExec_t> graphs;
  int smem_optin = 48 * 1024;  // opt-in dynamic shared memory per CTA on this device
};

namespace {

template <class T>
g4_status dalloc(g4_handle* h, T** p, size_t count) {
  void* q = nullptr;
  const size_t nbytes = std::max<size_t>(count, 1) * sizeof(T);
  if (h->fail_at > 0 && ++h->n_allocs == h->fail_at) return G4_ERR_OOM;  // injected
  cudaError_t e = cudaMalloc(&q, nbytes);
  if (e != cudaSuccess) {
    cuda_ok(e, "cudaMalloc");
    return e == cudaErrorMemoryAllocation ? G4_ERR_OOM : G4_ERR_CUDA;
  }
  h->allocs.push_back(q);
  h->bytes += nbytes;
  *p = reinterpret_cast<T*>(q);
  return G4_OK;
}
#define TRY(x)                          \
  do {                                  \
    g4_status s_ = (x);                 \
    if (s_ != G4_OK) return s_;         \
  } while (0)

int sgk(int fmt) { return fmt == G4_W4A16 ? Fmt<FMT_W4A16>::SGK : Fmt<FMT_BF16>::SGK; }

// Choose the per-CTA K chunk: enough CTAs to cover the SMs a few times, fewer, fatter CTAs
// for very tall matrices.
// Projections whose tiles take fewer bytes than this run with one K slice (no partial sums and
// no last-CTA merge on their dependency chain); 0 (the default) splits every projection.
// Environment G4_GEMV_UNSPLIT_BYTES, read once.
size_t gemv_unsplit_bytes() {
  static const size_t v = [] {
    const char* e = getenv("G4_GEMV_UNSPLIT_BYTES");
    return e ? (size_t)std::max(0LL, atoll(e)) : (size_t)0;
  }();
  return v;
}

void plan_lin(Lin& L, int sms, bool whole_k) {
  const int n_rg = L.n_rb / L.R;
  // start at one supergroup per CTA, halve the split while the grid exceeds 3 CTAs per SM; the
  // K slices are balanced (warps share a slice's tiles, whatever its supergroup count)
  int ks = (whole_k || L.bytes < gemv_unsplit_bytes()) ? 1 : L.S;
  while (ks > 1 && (long)n_rg * ks > 3L * sms) ks = cdiv(ks, 2);
  L.sg_per_cta = cdiv(L.S, ks);
  L.ksplit = cdiv(L.S, L.sg_per_cta);
}

// Build one tiled projection from row segments (each a multiple of 32 rows, except the
// last block of a single-segment matrix).  interleave: segments {gate, up} alternate
// 32-row blocks (R = 2) for the GeGLU epilogue.
g4_status build_lin(g4_handle* h, int fmt, int K, const std::vector<Seg>& segs, bool interleave, Lin* out,
                    cudaStream_t st, std::vector<RbSrc>& staging_keepalive) {
  Lin L;
  L.fmt = fmt;
  L.K = K;
  L.R = interleave ? 2 : 1;
  std::vector<RbSrc> rbs;
  const size_t rowbytes_w = fmt == G4_W4A16 ? (size_t)K / 2 : (size_t)K * 2;
  const size_t rowbytes_s = (size_t)K / 32 * 2;
  auto seg_blocks = [&](const Seg& s, std::vector<RbSrc>& v) {
    for (int r0 = 0; r0 < s.rows; r0 += 32) {
      RbSrc b;
      b.w = static_cast<const char*>(s.w) + r0 * rowbytes_w;
      b.s = s.s ? static_cast<const char*>(s.s) + r0 * rowbytes_s : nullptr;
      b.rows = std::min(32, s.rows - r0);
      b.pad = 0;
      v.push_back(b);
    }
  };
  if (interleave) {
    std::vector<RbSrc> g, u;
    seg_blocks(segs[0], g);
    seg_blocks(segs[1], u);
    for (size_t i = 0; i < g.size(); ++i) { rbs.push_back(g[i]); rbs.push_back(u[i]); }
    L.n_valid = segs[0].rows;
  } else {
    int n = 0;
    for (const Seg& s : segs) { seg_blocks(s, rbs); n += s.rows; }
    L.n_valid = n;
  }
  while (rbs.size() % 4) rbs.push_back(RbSrc{nullptr, nullptr, 0, 0});  // M tiles of 128 rows
  L.n_rb = (int)rbs.size();
  L.N = L.n_rb * 32;
  L.S = cdiv(K, sgk(fmt));
  L.tiles = 8 * L.S;
  TRY(dalloc(h, &L.qw, (size_t)L.n_rb * L.tiles * 32));
  L.bytes = (size_t)L.n_rb * L.tiles * 32 * 16;
  if (fmt == G4_W4A16) {
    TRY(dalloc(h, &L.sc, (size_t)L.n_rb * L.S * 32));
    L.bytes += (size_t)L.n_rb * L.S * 32 * 16;
  }
  RbSrc* d_rbs = nullptr;
  CK(cudaMalloc(&d_rbs, rbs.size() * sizeof(RbSrc)));
  cudaError_t e = cudaMemcpy(d_rbs, rbs.data(), rbs.size() * sizeof(RbSrc), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) {
    const int blocks = 4 * h->sms;
    if (fmt == G4_W4A16) {
      repack_int4_kernel<<<blocks, 256, 0, st>>>(d_rbs, L.n_rb, K, L.tiles, L.qw);
      repack_scales_kernel<<<blocks, 256, 0, st>>>(d_rbs, L.n_rb, K, L.S, L.sc);
    } else {
      repack_bf16_kernel<<<blocks, 256, 0, st>>>(d_rbs, L.n_rb, K, L.tiles, L.qw);
    }
    e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  cudaFree(d_rbs);
  CK(e);
  (void)staging_keepalive;
  *out = L;
  return G4_OK;
}

// ---------------------------------------------------------------------------- GEMV launch
struct GemvIO {
  int pro = PRO_PLAIN;
  const float* x_in = nullptr;
  int x_stride = 0;
  const float* r_in = nullptr;
  int r_stride = 0;
  int r_parts = 1;
  long r_part_stride = 0;
  const __nv_bfloat16* g_r = nullptr;
  float lambda = 1.f;
  const __nv_bfloat16* g_a = nullptr;
  float* x_out = nullptr;
  int norm_n = 0;
  float* y = nullptr;
  int y_stride = 0;
  const float* ple = nullptr;
  int ple_stride = 0;
  float* logits = nullptr;
  int logits_stride = 0;
  int* next_ids = nullptr;
};

struct Scratch {
  float* part;
  unsigned* cnt;
  float* am_val;
  int* am_idx;
  int* err;
};

// Programmatic dependent launch for every kernel of the step (G4_PDL=0 disables it).
bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("G4_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
void launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaLaunchKernelEx(&cfg, kern, args...);
}

// Every kernel of a step prefers the largest shared-memory carve-out.  Under programmatic
// dependent launch the next kernel's CTAs become resident while the current kernel runs and
// stream their weights in; an SM configured for a smaller carve-out can take a CTA that needs
// more shared memory only after it drains, which delays that CTA (and its weight loads) to
// the end of the current kernel.  With one carve-out for all kernels any mix of CTAs fits.
template <typename... KArgs>
void carve_max(void (*k)(KArgs...)) {
  cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
}
// Opt every kernel into the full shared-memory carve-out once per process (never during a
// stream capture).
template <typename... KArgs>
void set_max_dyn(void (*k)(KArgs...), int optin) {
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) return;
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
  carve_max(k);
}
template <int FMT, int R, int EPI>
void attrs_gemv(int optin) {
  set_max_dyn(gemv_kernel<FMT, R, 1, EPI>, optin);
  set_max_dyn(gemv_kernel<FMT, R, 2, EPI>, optin);
  set_max_dyn(gemv_kernel<FMT, R, 4, EPI>, optin);
}
template <int FMT>
void attrs_staged(int optin) {
  set_max_dyn(gemv_s_kernel<FMT, 1, 1, EPI_STORE>, optin);
  set_max_dyn(gemv_s_kernel<FMT, 1, 2, EPI_STORE>, optin);
  set_max_dyn(gemv_s_kernel<FMT, 1, 4, EPI_STORE>, optin);
  set_max_dyn(gemv_s_kernel<FMT, 1, 1, EPI_ARGMAX>, optin);
  set_max_dyn(gemv_s_kernel<FMT, 1, 2, EPI_ARGMAX>, optin);
  set_max_dyn(gemv_s_kernel<FMT, 1, 4, EPI_ARGMAX>, optin);
}
template <int D>
void attrs_attn(int optin) {
  set_max_dyn(attn_mqa_kernel<D, false>, optin);
  set_max_dyn(attn_mqa_kernel<D, true>, optin);
  set_max_dyn(attn_kernel<D, 1, false>, optin);
  set_max_dyn(attn_kernel<D, 1, true>, optin);
  carve_max(kv_write_kernel<D, false>);
  carve_max(kv_write_kernel<D, true>);
}
std::mutex g_attr_mu;
std::map<int, int> g_optin;  // device -> opt-in shared memory bytes
int init_kernel_attrs(int device) {
  std::lock_guard<std::mutex> lk(g_attr_mu);
  auto it = g_optin.find(device);
  if (it != g_optin.end()) return it->second;
  int optin = 48 * 1024;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  attrs_gemv<FMT_W4A16, 1, EPI_STORE>(optin);
  attrs_gemv<FMT_BF16, 1, EPI_STORE>(optin);
  attrs_gemv<FMT_W4A16, 2, EPI_GEGLU>(optin);
  attrs_gemv<FMT_BF16, 2, EPI_GEGLU>(optin);
  attrs_gemv<FMT_W4A16, 1, EPI_PLE>(optin);
  attrs_gemv<FMT_BF16, 1, EPI_PLE>(optin);
  attrs_gemv<FMT_BF16, 1, EPI_ARGMAX>(optin);
  attrs_gemv<FMT_W4A16, 1, EPI_ARGMAX>(optin);
  attrs_staged<FMT_W4A16>(optin);
  attrs_staged<FMT_BF16>(optin);
  set_max_dyn(gemm_tc_kernel, optin);
  set_max_dyn(mega_step_kernel<1>, optin);
  set_max_dyn(mega_step_kernel<2>, optin);
  set_max_dyn(prep_x_kernel, optin);
  attrs_attn<64>(optin);
  attrs_attn<128>(optin);
  attrs_attn<256>(optin);
  attrs_attn<512>(optin);
  carve_max(embed_kernel);
  carve_max(ple_combine_kernel);
  carve_max(gather_rows_kernel);
  carve_max(argmax_partials_kernel);
  cudaGetLastError();
  g_optin[device] = optin;
  return optin;
}

template <int FMT, int R, int EPI>
void launch_fmt(const GemvArgs& a, int nb, int grid, cudaStream_t st) {
  const int kc = a.sg_per_cta * Fmt<FMT>::SGK;
  if (nb == 1) {
    const size_t sm = gemv_smem_plan(1, R, kc, a.pro, a.norm_n, a.ksplit).total_floats * 4;
    launch(gemv_kernel<FMT, R, 1, EPI>, dim3(grid), dim3(kGemvThreads), sm, st, a);
  } else if (nb == 2) {
    const size_t sm = gemv_smem_plan(2, R, kc, a.pro, a.norm_n, a.ksplit).total_floats * 4;
    launch(gemv_kernel<FMT, R, 2, EPI>, dim3(grid), dim3(kGemvThreads), sm, st, a);
  } else {
    const size_t sm = gemv_smem_plan(4, R, kc, a.pro, a.norm_n, a.ksplit).total_floats * 4;
    launch(gemv_kernel<FMT, R, 4, EPI>, dim3(grid), dim3(kGemvThreads), sm, st, a);
  }
}

// Grid of one GEMV launch: every (row group, K slice) when split; otherwise persistent CTAs
// (at most 4 per SM) looping over row groups.
int gemv_grid(const Lin& L, int sms) {
  const int n_rg = L.n_rb / L.R;
  if (L.ksplit > 1) return n_rg * L.ksplit;
  return std::min(n_rg, 4 * sms);
}

// ------------------------------------------------------------------- staged GEMV launch
// The staged projection (gemv_s.cuh) runs every projection of a decode step of 1-4 rows but
// the lm_head; the environment G4_GEMV_STAGED=0 sends them to the K-split GEMV instead (for
// comparisons).
bool gemv_staged_on() {
  static const bool on = [] {
    const char* e = getenv("G4_GEMV_STAGED");
    return !(e && e[0] == '0');
  }();
  return on;
}

constexpr int kSgSmemBudget = 110 * 1024;  // CTAs of two consecutive launches share an SM
constexpr int kSgCtrSlots = 512;           // staged launches of one step (row-group counters)

// Partition of one projection over the SMs: C K slices (C = 1 when the epilogue needs whole
// sums), floor(sms / C) * C CTAs, row blocks taken one at a time.  Chooses C to minimise the
// tiles the busiest CTA streams, ceil(row blocks / CTAs per slice) x slice, counting 4 tiles
// per row block taken (its sums) and 8 per extra part the consumer adds; ties go to fewer
// slices.  Then ring items of up to 32 KB and as many ring slots as the shared-memory budget
// allows.
struct SPlan {
  bool ok = false;
  GemvSArgs a{};
  size_t smem = 0;
  int grid = 0;
};
SPlan plan_staged(const Lin& L, int NB, int pro, int norm_n, bool whole_sums, int sms) {
  SPlan p;
  const bool w4 = L.fmt == G4_W4A16;
  const int sgb = 8 * 512 + (w4 ? 512 : 0);
  const int sg_k = sgk(L.fmt);
  const int n_rb = L.n_rb;  // units: single row blocks (R = 1)
  long best = -1;
  for (int C = 1; C <= kSgMaxParts && C <= L.S; ++C) {
    if (whole_sums && C > 1) break;
    const int spc = cdiv(L.S, C);
    if (cdiv(L.S, spc) != C) continue;  // every slice non-empty
    const int per = sms / C;            // CTAs per slice
    if (per < 1) break;
    const int rounds = cdiv(n_rb, per);
    const int cap = std::min(kSgMaxUnits, 2 * rounds + 1);
    if ((long)cap * per < n_rb) continue;
    const long cost = (long)rounds * (spc * 8 + 4) + 8L * (C - 1);
    if (best < 0 || cost < best) {
      best = cost;
      p.a.C = C;
      p.a.spc = spc;
      p.a.cap = cap;
      p.a.ru = cap;
      p.grid = per * C;
    }
  }
  if (best < 0) return p;
  GemvSArgs& a = p.a;
  a.csg = std::max(1, std::min({a.spc, kSgMaxCsg, 32768 / sgb}));
  a.slot_bytes = (a.csg * sgb + 127) / 128 * 128;
  a.pro = pro;
  a.norm_n = norm_n;
  a.slots = std::min(kSgMaxSlots, a.cap * cdiv(a.spc, a.csg) + 1);
  for (;;) {
    const SgSmem m = sg_smem_plan(NB, 1, sg_k, a);
    p.smem = (size_t)m.total + 128;
    if ((int)p.smem <= kSgSmemBudget || a.slots <= 2) break;
    --a.slots;
  }
  p.ok = (int)p.smem <= kSgSmemBudget + 64 * 1024;
  return p;
}

// One CTA per SM for every staged launch.  Consecutive launches share SMs (the next one streams
// its weights while the current one computes), so each CTA takes a little under half of an SM;
// with nothing else in the way, the CTA scheduler then puts two CTAs of ONE launch on an SM
// wherever the previous launch left a hole, and such an SM runs both at half speed.  A wide
// attention launch (more CTAs than SMs) made those holes, and they carried over from launch to
// launch for the rest of the step.  The step therefore alternates two footprints:
//   X: dynamic shared memory padded past half an SM (two X CTAs cannot share an SM);
//   Y: padding warps that take the CTA's registers past half the register file (two Y CTAs
//      cannot share one), with shared memory within the budget;
// an X CTA and a Y CTA fit together (96 registers a thread by construction).
constexpr int kSgSmemPerSm = 228 * 1024;     // shared memory of one SM
constexpr int kSgSmemPerCta = 1024;          // reserved by the system per resident CTA
constexpr int kSgXSmem = kSgSmemPerSm / 2 - kSgSmemPerCta + 2048;   // > half an SM with the reserve
static_assert(2 * (kSgXSmem + kSgSmemPerCta) > kSgSmemPerSm, "X footprint must exceed half an SM");
static_assert((kSgXSmem + kSgSmemPerCta) + (kSgSmemBudget + kSgSmemPerCta) <= kSgSmemPerSm,
              "X and Y footprints must fit together");
template <typename K>
int staged_y_threads(K kernel) {
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess || fa.numRegs <= 0) return kSgThreads;
  const int r = (fa.numRegs + 7) / 8 * 8;           // allocation granularity
  const int warps = std::max(kSgWarps + 2, 65536 / 2 / (32 * r) + 1);
  // X (kSgThreads at r <= kSgMaxRegs) beside Y must still fit the register file
  if (kSgThreads * kSgMaxRegs + warps * 32 * r > 65536) return kSgThreads;
  return warps * 32;
}
template <int FMT, int NB>
void launch_staged_nb(const GemvSArgs& a, int grid, size_t smem, int xy, cudaStream_t st) {
  static const int y_threads = staged_y_threads(gemv_s_kernel<FMT, 1, NB, EPI_STORE>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(xy == 2 ? y_threads : kSgThreads);
  if (xy == 1) smem = std::max(smem, (size_t)kSgXSmem);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaLaunchKernelEx(&cfg, gemv_s_kernel<FMT, 1, NB, EPI_STORE>, a);
}

// Input of a staged projection (see gemv_s.cuh).  The residual branch and the PRO_GEGLU /
// PRO_PLEG sources may come as `parts` K-slice partial sums, part q at base + q * part_stride.
struct StagedIn {
  int pro = PRO_PLAIN;
  const float* x = nullptr;
  int x_stride = 0;
  int x_parts = 1;
  long x_part_stride = 0;
  const float* r = nullptr;
  int r_stride = 0;
  int r_parts = 1;
  long r_part_stride = 0;
  const __nv_bfloat16* g_r = nullptr;
  float lambda = 1.f;
  const __nv_bfloat16* g_a = nullptr;
  float* x_out = nullptr;
  const float* ple = nullptr;  // PRO_PLEG: multiplier rows
  int ple_stride = 0;
};
// Output of a staged projection: raw sums, part c at y + c * part_stride.  `parts` receives C.
struct StagedOut {
  float* y = nullptr;
  int y_stride = 0;
  long part_stride = 0;
  int* parts = nullptr;
};

// y = W x (raw K-slice partial sums; with whole_sums one slice, so y is the product) through
// the staged kernel.  ctr: this launch's row-group counters ([2][kSgMaxParts], zero).  False if
// the projection has no staged plan.
// xy: 0 plain launch, 1 / 2 the X / Y footprint (above).
bool run_staged(const Lin& L, const StagedIn& in, const StagedOut& out, int n, float eps, int* err, unsigned* ctr,
                int sms, cudaStream_t st, bool whole_sums = false, int xy = 0) {
  const int NB = n == 1 ? 1 : (n == 2 ? 2 : 4);
  const int norm_n = (in.pro == PRO_NORM || in.pro == PRO_RESID) ? L.K : 0;
  SPlan p = plan_staged(L, NB, in.pro, norm_n, whole_sums, sms);
  if (!p.ok) return false;
  GemvSArgs& a = p.a;
  a.qw = L.qw;
  a.sc = L.sc;
  a.n_rb = L.n_rb;
  a.S = L.S;
  a.tiles = L.tiles;
  a.K = L.K;
  a.n_valid = L.R == 2 ? 2 * L.n_valid : L.n_valid;  // raw rows: both halves of an interleaved pair
  a.grab = ctr;
  a.done = ctr + kSgMaxParts;
  a.nb = n;
  a.x_in = in.x;
  a.x_stride = in.x_stride;
  a.x_parts = in.x_parts;
  a.x_part_stride = in.x_part_stride;
  a.r_in = in.r;
  a.r_stride = in.r_stride;
  a.r_parts = in.r_parts;
  a.r_part_stride = in.r_part_stride;
  a.g_r = in.g_r;
  a.lambda = in.lambda;
  a.g_a = in.g_a;
  a.x_out = in.x_out;
  a.eps = eps;
  a.y = out.y;
  a.y_stride = out.y_stride;
  a.y_part_stride = out.part_stride;
  a.ple = in.ple;
  a.ple_stride = in.ple_stride;
  a.err = err;
  if (out.parts) *out.parts = a.C;
  if ((int)p.smem > kSgSmemBudget) xy = 0;  // the footprints assume the budget
  const bool w4 = L.fmt == G4_W4A16;
  if (NB == 1) w4 ? launch_staged_nb<FMT_W4A16, 1>(a, p.grid, p.smem, xy, st) : launch_staged_nb<FMT_BF16, 1>(a, p.grid, p.smem, xy, st);
  else if (NB == 2) w4 ? launch_staged_nb<FMT_W4A16, 2>(a, p.grid, p.smem, xy, st) : launch_staged_nb<FMT_BF16, 2>(a, p.grid, p.smem, xy, st);
  else w4 ? launch_staged_nb<FMT_W4A16, 4>(a, p.grid, p.smem, xy, st) : launch_staged_nb<FMT_BF16, 4>(a, p.grid, p.smem, xy, st);
  return true;
}

// The vocabulary projection with the greedy choice (EPI_ARGMAX of gemv_s.cuh) on the staged
// kernel: one K slice, one CTA per SM taking row blocks until none is left, and as many ring
// slots as the opt-in shared memory holds (it is the step's last kernel and the longest
// stream: the more weight bytes in flight per SM, the closer to the HBM rate).  By default it
// takes the W4A16 vocabulary table (E2B, batch 1: 226 MB in place of the GEMV's three CTAs
// per SM at 160 registers); a bf16 table stays on the persistent GEMV, which streamed it
// faster.  The environment G4_LMHEAD_STAGED=0 keeps both on the GEMV, =1 puts both on the
// staged kernel (for comparisons).
bool lmhead_staged(int fmt) {
  static const int mode = [] {
    const char* e = getenv("G4_LMHEAD_STAGED");
    return e ? (e[0] == '0' ? 0 : 1) : 2;
  }();
  return mode == 1 || (mode == 2 && fmt == G4_W4A16);
}
SPlan plan_staged_argmax(const Lin& L, int NB, int norm_n, int sms, int smem_max) {
  SPlan p;
  const bool w4 = L.fmt == G4_W4A16;
  const int sgb = 8 * 512 + (w4 ? 512 : 0);
  GemvSArgs& a = p.a;
  a.C = 1;
  a.spc = L.S;
  a.cap = L.n_rb;
  a.am = 1;
  a.csg = std::max(1, std::min({a.spc, kSgMaxCsg, 32768 / sgb}));
  a.slot_bytes = (a.csg * sgb + 127) / 128 * 128;
  a.pro = PRO_RESID;
  a.norm_n = norm_n;
  const int nch = cdiv(a.spc, a.csg);
  for (a.slots = kSgMaxSlots;; --a.slots) {
    a.ru = cdiv(a.slots, nch) + 2;  // ru * nch > slots + nch: a unit slot is free when reused
    p.smem = (size_t)sg_smem_plan(NB, 1, sgk(L.fmt), a).total + 128;
    if ((int)p.smem <= smem_max || a.slots <= 2) break;
  }
  p.grid = sms;
  p.ok = (int)p.smem <= smem_max && a.ru <= kSgMaxUnits && a.slots >= 2;
  return p;
}
template <int FMT, int NB>
void launch_staged_argmax_nb(const GemvSArgs& a, int grid, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSgThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaLaunchKernelEx(&cfg, gemv_s_kernel<FMT, 1, NB, EPI_ARGMAX>, a);
}
// logits = W x (optional, [n][logits_stride]) and next_ids[b] = argmax_n logits[b][n] for the
// residual-prologue input `in`.  am_val / am_idx: n * sms entries; am_cnt: zero, left zero.
// False if the projection has no such plan (the caller uses the GEMV).
bool run_staged_argmax(const Lin& L, const StagedIn& in, float* logits, int logits_stride, int* next_ids, int n,
                       float eps, int* err, unsigned* ctr, float* am_val, int* am_idx, unsigned* am_cnt, int sms,
                       int smem_max, cudaStream_t st) {
  if (L.R != 1 || in.pro != PRO_RESID || n < 1 || n > kMaxNB) return false;
  const int NB = n == 1 ? 1 : (n == 2 ? 2 : 4);
  SPlan p = plan_staged_argmax(L, NB, L.K, sms, smem_max);
  if (!p.ok) return false;
  GemvSArgs& a = p.a;
  a.qw = L.qw;
  a.sc = L.sc;
  a.n_rb = L.n_rb;
  a.S = L.S;
  a.tiles = L.tiles;
  a.K = L.K;
  a.n_valid = L.n_valid;
  a.grab = ctr;
  a.done = ctr + kSgMaxParts;
  a.nb = n;
  a.x_in = in.x;
  a.x_stride = in.x_stride;
  a.x_parts = 1;
  a.r_in = in.r;
  a.r_stride = in.r_stride;
  a.r_parts = in.r_parts;
  a.r_part_stride = in.r_part_stride;
  a.g_r = in.g_r;
  a.lambda = in.lambda;
  a.g_a = in.g_a;
  a.x_out = in.x_out;
  a.eps = eps;
  a.y = logits;
  a.y_stride = logits_stride;
  a.err = err;
  a.am_val = am_val;
  a.am_idx = am_idx;
  a.am_cnt = am_cnt;
  a.next_ids = next_ids;
  const bool w4 = L.fmt == G4_W4A16;
  if (NB == 1) w4 ? launch_staged_argmax_nb<FMT_W4A16, 1>(a, p.grid, p.smem, st) : launch_staged_argmax_nb<FMT_BF16, 1>(a, p.grid, p.smem, st);
  else if (NB == 2) w4 ? launch_staged_argmax_nb<FMT_W4A16, 2>(a, p.grid, p.smem, st) : launch_staged_argmax_nb<FMT_BF16, 2>(a, p.grid, p.smem, st);
  else w4 ? launch_staged_argmax_nb<FMT_W4A16, 4>(a, p.grid, p.smem, st) : launch_staged_argmax_nb<FMT_BF16, 4>(a, p.grid, p.smem, st);
  return true;
}

// Tensor-core path for batches >= G4_TC_MIN_BATCH (default 5; 0 disables it).  The GEMV
// takes up to kMaxNB = 4 rows per launch; from 5 rows it would need a second pass, and the
// tensor-core step measured faster (E2B W4A16, batch 8: 4.27 against 8.72 ms per step).
int tc_min_batch() {
  static const int v = [] {
    const char* e = getenv("G4_TC_MIN_BATCH");
    return e ? atoi(e) : 5;
  }();
  return v;
}
int tc_bpad(int n) { return (n + 15) / 16 * 16; }
int tc_nkb(const Lin& L) { return cdiv(L.K, kTcKB); }
// K split so that M tiles x splits roughly fill the SMs once (one CTA per SM).
void tc_plan(const Lin& L, int sms, bool whole_k, int* ksplit, int* kbps) {
  const int nmt = L.n_rb / 4, nkb = tc_nkb(L);
  // at least 4 k-blocks per split: the split-K reduction is not free
  // and at most 6 splits: the last CTA's merge costs a few L2 round trips per 3 splits
  int k = whole_k ? 1 : std::max(1, std::min({cdiv(nkb, 4), sms / std::max(1, nmt), 6}));
  *kbps = cdiv(nkb, k);
  *ksplit = cdiv(nkb, *kbps);
}

struct TcScratch {
  uint8_t* xt;
  float* part;
  unsigned* cnt;
  float* am_val;
  int* am_idx;
  int* err;
};

void run_gemm(const Lin& L, int epi, const GemvIO& io, int n, float eps, const TcScratch& s, int sms, cudaStream_t st) {
  const int bpad = tc_bpad(n), nkb = tc_nkb(L);
  PrepArgs p{};
  p.pro = io.pro;
  p.x_in = io.x_in;
  p.x_stride = io.x_stride;
  p.r_in = io.r_in;
  p.r_stride = io.r_stride;
  p.g_r = io.g_r;
  p.lambda = io.lambda;
  p.g_a = io.g_a;
  p.x_out = io.x_out;
  p.eps = eps;
  p.K = L.K;
  p.kpad = nkb * kTcKB;
  p.bpad = bpad;
  p.xt = s.xt;
  launch(prep_x_kernel, dim3(n), dim3(256), prep_smem_bytes(p.kpad, p.pro), st, p);
  GemmArgs g{};
  g.qw = L.qw;
  g.sc = L.sc;
  g.fmt = L.fmt == G4_W4A16 ? FMT_W4A16 : FMT_BF16;
  g.tiles = L.tiles;
  g.S = L.S;
  g.n_valid = L.n_valid;
  g.n_kb = nkb;
  tc_plan(L, sms, epi == EPI_ARGMAX, &g.ksplit, &g.kb_per_split);
  g.xt = s.xt;
  g.bpad = bpad;
  g.nb = n;
  g.epi = epi;
  g.y = io.y;
  g.y_stride = io.y_stride;
  g.ple = io.ple;
  g.ple_stride = io.ple_stride;
  g.logits = io.logits;
  g.logits_stride = io.logits_stride;
  g.am_val = s.am_val;
  g.am_idx = s.am_idx;
  g.part = s.part;
  g.counters = s.cnt;
  g.n_mtiles = L.n_rb / 4;
  g.err = s.err;
  const int grid = g.n_mtiles * g.ksplit;
  g.stages = g.ksplit > 1 ? kTcStages : 2;
  launch(gemm_tc_kernel, dim3(grid), dim3(kTcThreads), tc_smem_bytes(bpad, g.stages), st, g);
  if (epi == EPI_ARGMAX)
    launch(argmax_partials_kernel, dim3(n), dim3(256), 0, st, (const float*)s.am_val, (const int*)s.am_idx, grid,
           io.next_ids);
}

// y = W x for n rows, in chunks of kMaxNB rows.
void run_gemv(const Lin& L, int epi, const GemvIO& io, int n, float eps, const Scratch& s, int sms,
              cudaStream_t st, const TcScratch* tc = nullptr) {
  if (tc && tc_min_batch() > 0 && n >= tc_min_batch() && n <= 64) {
    run_gemm(L, epi, io, n, eps, *tc, sms, st);
    return;
  }
  for (int b0 = 0; b0 < n; b0 += kMaxNB) {
    const int nb = std::min(kMaxNB, n - b0);
    GemvArgs a{};
    a.qw = L.qw;
    a.sc = L.sc;
    a.n_rb = L.n_rb;
    a.n_valid = L.n_valid;
    a.K = L.K;
    a.S = L.S;
    a.tiles = L.tiles;
    a.nb = nb;
    a.ksplit = L.ksplit;
    a.sg_per_cta = L.sg_per_cta;
    a.pro = io.pro;
    a.x_in = io.x_in + (size_t)b0 * io.x_stride;
    a.x_stride = io.x_stride;
    a.r_in = io.r_in ? io.r_in + (size_t)b0 * io.r_stride : nullptr;
    a.r_stride = io.r_stride;
    a.r_parts = io.r_parts;
    a.r_part_stride = io.r_part_stride;
    a.g_r = io.g_r;
    a.lambda = io.lambda;
    a.g_a = io.g_a;
    a.x_out = io.x_out ? io.x_out + (size_t)b0 * io.x_stride : nullptr;
    a.eps = eps;
    a.norm_n = io.norm_n;
    a.y = io.y ? io.y + (size_t)b0 * io.y_stride : nullptr;
    a.y_stride = io.y_stride;
    a.ple = io.ple ? io.ple + (size_t)b0 * io.ple_stride : nullptr;
    a.ple_stride = io.ple_stride;
    a.logits = io.logits ? io.logits + (size_t)b0 * io.logits_stride : nullptr;
    a.logits_stride = io.logits_stride;
    a.am_val = s.am_val;
    a.am_idx = s.am_idx;
    a.next_ids = io.next_ids ? io.next_ids + b0 : nullptr;
    a.part = s.part;
    a.counters = s.cnt;
    const int grid = gemv_grid(L, sms);
    const bool w4 = L.fmt == G4_W4A16;
    switch (epi) {
      case EPI_STORE:
        if (w4) launch_fmt<FMT_W4A16, 1, EPI_STORE>(a, nb, grid, st);
        else launch_fmt<FMT_BF16, 1, EPI_STORE>(a, nb, grid, st);
        break;
      case EPI_GEGLU:
        if (w4) launch_fmt<FMT_W4A16, 2, EPI_GEGLU>(a, nb, grid, st);
        else launch_fmt<FMT_BF16, 2, EPI_GEGLU>(a, nb, grid, st);
        break;
      case EPI_PLE:
        if (w4) launch_fmt<FMT_W4A16, 1, EPI_PLE>(a, nb, grid, st);
        else launch_fmt<FMT_BF16, 1, EPI_PLE>(a, nb, grid, st);
        break;
      case EPI_ARGMAX:
        if (w4) launch_fmt<FMT_W4A16, 1, EPI_ARGMAX>(a, nb, grid, st);
        else launch_fmt<FMT_BF16, 1, EPI_ARGMAX>(a, nb, grid, st);
        break;
    }
  }
}

// ---------------------------------------------------------------------- attention launch
template <int D, int HPC, bool KV8>
void launch_attn(const AttnArgs& a, int nb, cudaStream_t st) {
  dim3 grid(a.nsplit, a.nq / HPC, nb);
  launch(attn_kernel<D, HPC, KV8>, grid, dim3(kAttnThreads), attn_smem_bytes<D, HPC, KV8>(a.nstage), st, a);
}
template <int D>
void launch_attn_d(const AttnArgs& a, int hpc, int nb, bool kv8, cudaStream_t st) {
  (void)hpc;  // attn_hpc: one head per unit
  if (kv8) launch_attn<D, 1, true>(a, nb, st);
  else launch_attn<D, 1, false>(a, nb, st);
}
template <int D, bool KV8>
void launch_mqa(const AttnArgs& a, int nb, cudaStream_t st) {
  launch(attn_mqa_kernel<D, KV8>, dim3(a.nsplit, nb), dim3(kMqaThreads), mqa_smem_bytes<D, KV8>(a.nstage), st, a);
}
template <int D>
void launch_mqa_d(const AttnArgs& a, int nb, bool kv8, cudaStream_t st) {
  if (kv8) launch_mqa<D, true>(a, nb, st);
  else launch_mqa<D, false>(a, nb, st);
}
// mqa: the kernel that serves every query head of a sequence from one K/V tile load
// (attn_mqa.cuh); else one CTA per (split, head) (attn.cuh).
void launch_attn_any(const AttnArgs& a, int d, int hpc, int nb, bool kv8, bool mqa, cudaStream_t st) {
  if (mqa) {
    switch (d) {
      case 64: launch_mqa_d<64>(a, nb, kv8, st); break;
      case 128: launch_mqa_d<128>(a, nb, kv8, st); break;
      case 256: launch_mqa_d<256>(a, nb, kv8, st); break;
      default: launch_mqa_d<512>(a, nb, kv8, st); break;
    }
    return;
  }
  switch (d) {
    case 64: launch_attn_d<64>(a, hpc, nb, kv8, st); break;
    case 128: launch_attn_d<128>(a, hpc, nb, kv8, st); break;
    case 256: launch_attn_d<256>(a, hpc, nb, kv8, st); break;
    default: launch_attn_d<512>(a, hpc, nb, kv8, st); break;
  }
}
template <int D>
void launch_kv_write_d(const AttnArgs& a, int nb, bool kv8, cudaStream_t st) {
  if (kv8) launch(kv_write_kernel<D, true>, dim3(nb), dim3(32), 0, st, a);
  else launch(kv_write_kernel<D, false>, dim3(nb), dim3(32), 0, st, a);
}
void launch_kv_write_any(const AttnArgs& a, int d, int nb, bool kv8, cudaStream_t st) {
  switch (d) {
    case 64: launch_kv_write_d<64>(a, nb, kv8, st); break;
    case 128: launch_kv_write_d<128>(a, nb, kv8, st); break;
    case 256: launch_kv_write_d<256>(a, nb, kv8, st); break;
    default: launch_kv_write_d<512>(a, nb, kv8, st); break;
  }
}

// Query heads per attention unit.  One: a unit per (split, head, sequence) keeps every unit's
// dependency chain short; at batch 64 this measured faster than eight heads per unit (which
// share one K/V tile load but serialise eight heads' scores and outputs in one CTA).
int attn_hpc(int nq, int nb) {
  (void)nq;
  (void)nb;
  return 1;
}
// Tokens per prefill block: one step over the rows of a prompt (the tensor-core GEMMs take up
// to 64 rows).
constexpr int kPrefillRows = 64;

int attn_nsplit(int sms, int nq, int hpc, int nb, int max_keys) {
  const int n_hg = nq / hpc;
  int ns = cdiv(2 * sms, nb * n_hg);
  ns = std::min(ns, std::max(1, cdiv(max_keys, kAttnTile)));
  return std::max(1, std::min(ns, 64));
}
// The MQA kernel: one CTA per (split, sequence); about two per SM.
int mqa_nsplit(int sms, int nb, int max_keys) {
  int ns = cdiv(2 * sms, nb);
  ns = std::min(ns, std::max(1, cdiv(max_keys, kAttnTile)));
  return std::max(1, std::min(ns, 64));
}
// From this many sequences on, attention runs the MQA kernel (G4_ATTN_MQA_MIN; 0 disables
// it).  Below, one CTA per (split, head) keeps a single sequence's latency short: the MQA
// kernel has fewer CTAs to spread one sequence's keys over and a longer merge.
int mqa_min_batch() {  // read at every plan (a graph keeps the choice it was captured with)
  const char* e = getenv("G4_ATTN_MQA_MIN");
  return e ? atoi(e) : 8;
}
bool mqa_on(int nq, int n) { return mqa_min_batch() > 0 && n >= mqa_min_batch() && nq <= kMqaMaxHeads; }
// Splits and tile buffers of an attention launch over n sequences (either kernel).
void attn_plan(int sms, int nq, int n, int d, int max_keys, AttnArgs& a) {
  if (mqa_on(nq, n)) {
    a.nsplit = mqa_nsplit(sms, n, max_keys);
    a.nstage = (d <= 256 && cdiv(max_keys, a.nsplit) > kAttnTile) ? 2 : 1;
    return;
  }
  const int hpc = attn_hpc(nq, n);
  a.nsplit = attn_nsplit(sms, nq, hpc, n, max_keys);
  // double-buffered K/V tiles only while the grid fits on the SMs at one unit each: a
  // larger grid needs the occupancy more than the overlap (the 512-wide tiles take 128 KB)
  const long units = (long)n * (nq / hpc) * a.nsplit;
  a.nstage = (cdiv(max_keys, a.nsplit) > kAttnTile && units <= sms) ? 2 : 1;
}

// ------------------------------------------------------------------------------- profiler
// Optional CUDA-event bracketing of every launch of a (non-captured) step, by phase name.
struct Prof {
  struct Rec {
    std::string name;
    double bytes;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  cudaStream_t st = nullptr;
  void begin(const char* name, double bytes) {
    Rec r{name, bytes, nullptr, nullptr};
    cudaEventCreate(&r.a);
    cudaEventCreate(&r.b);
    cudaEventRecord(r.a, st);
    recs.push_back(r);
  }
  void end() { cudaEventRecord(recs.back().b, st); }
  ~Prof() {
    for (Rec& r : recs) { cudaEventDestroy(r.a); cudaEventDestroy(r.b); }
  }
};
struct ProfScope {
  Prof* p;
  ProfScope(Prof* p_, const char* name, double bytes) : p(p_) { if (p) p->begin(name, bytes); }
  ~ProfScope() { if (p) p->end(); }
};

// ------------------------------------------------------------------------------- the step
g4_status run_step_mega(g4_handle* h, cudaStream_t st, int n, const int* d_slots, const int* d_tokens,
                        const int* d_idx, const int* d_pos, int* d_next, float* d_logits, bool stamps);
// kv_first: write every row's K/V before the attention launch (prefill blocks, where rows of
// one sequence at consecutive positions attend to each other's keys).  n_keep >= 0: from the
// first layer after which no layer writes K/V on, only rows keep_idx[0 .. n_keep) (their
// slots and positions in keep_slots / keep_pos) go on: a prompt row that ends no sequence
// feeds nothing past its last K/V write.  n_keep == 0 ends the step there.
// int4 vocabulary tables in the embedding gather's arguments.
void set_tables(const g4_handle* h, EmbedArgs& ea) {
  ea.t4 = h->t4;
  ea.embed_q = h->embed_q;
  ea.embed_s = h->embed_s;
  ea.ple_q = h->ple_q;
  ea.ple_s = h->ple_s;
  ea.ple_group = h->cfg.ple_dim;
}
// Cache of layer Src (its K/V rows, scales and page table) in attention arguments.
void kv_args(const g4_handle* h, const Layer& Src, AttnArgs& a) {
  a.kc = h->kc[Src.kv];
  a.vc = h->vc[Src.kv];
  a.ksc = h->kv8 ? h->ksc[Src.kv] : nullptr;
  a.vsc = h->kv8 ? h->vsc[Src.kv] : nullptr;
  a.page_table = h->page_table;
  a.page_shift = h->page_shift;
  a.max_pages = h->max_pages;
}
// Attention launch of layer l (shared by both step paths).
void launch_layer_attn(g4_handle* h, const Layer& Y, const float* qkv, int qkv_stride, int n, const int* d_slots,
                       const int* d_pos, bool own, cudaStream_t st) {
  const g4_config& c = h->cfg;
  const Layer& Src = h->layers[Y.src];
  AttnArgs a{};
  a.qkv = qkv;
  a.qkv_stride = qkv_stride;
  a.nq = c.num_q_heads;
  a.g_q = Y.q_norm;
  a.g_k = Y.k_norm;
  a.eps = c.rms_eps;
  a.scale = Y.scale;
  a.window = Y.full ? 0 : c.sliding_window;
  a.own = own;
  a.early = 1;  // decode: no kernel right before writes cache rows
  kv_args(h, Src, a);
  a.t_max = c.max_context;
  a.max_batch = c.max_batch;
  a.rope_cos = h->cos_t[Y.full];
  a.rope_sin = h->sin_t[Y.full];
  a.slots = d_slots;
  a.positions = d_pos;
  a.out = h->attn;
  a.out_stride = c.num_q_heads * Y.d;
  const int hpc = attn_hpc(c.num_q_heads, n);
  const int max_keys = Y.full ? c.max_context : std::min(c.sliding_window, c.max_context);
  attn_plan(h->sms, c.num_q_heads, n, Y.d, max_keys, a);
  a.ws_ml = h->attn_ml;
  a.ws_o = h->attn_o;
  a.counters = h->attn_cnt;
  a.err = h->err;
  launch_attn_any(a, Y.d, hpc, n, h->kv8, mqa_on(c.num_q_heads, n), st);
}

// Decode step of 1-4 rows on the staged projections (gemv_s.cuh).  Every projection but the
// lm_head writes raw K-slice partial sums; the kernel that reads them adds the parts and applies
// what the projection's epilogue would have: the GeGLU (down's input), the per-layer-input gate
// (the per-layer projection's input), the residual update and norms (the next projection's
// prologue), the q/k/v split (attention), the per-layer-embedding combine.
g4_status run_step_staged(g4_handle* h, cudaStream_t st, int n, const int* d_slots, const int* d_tokens,
                          const int* d_idx, const int* d_pos, int* d_next, float* d_logits, Prof* prof) {
  const g4_config& c = h->cfg;
  const int H = c.hidden, L = c.num_layers, P = c.ple_dim, LP = L * P;
  const float eps = c.rms_eps;
  const long ps_h = (long)kMaxNB * H;  // part strides of the [part][row][width] buffers
  int seq = 0;                         // staged launches so far (their counter slots)
  auto ctr = [&]() { return h->sg_ctr + (size_t)(seq++ % kSgCtrSlots) * 2 * kSgMaxParts; };
  // whole: one K slice (attention reads q, k and v whole: its loads stay one round trip)
  auto staged = [&](const Lin& Ln, const StagedIn& in, float* y, int y_stride, long part_stride, int* parts,
                    const char* name, bool whole = false) -> g4_status {
    ProfScope ps(prof, name, (double)Ln.bytes);
    StagedOut out{y, y_stride, part_stride, parts};
    const int xy = (seq & 1) ? 2 : 1;  // consecutive staged launches alternate footprints
    if (!run_staged(Ln, in, out, n, eps, h->err, ctr(), h->sms, st, whole, xy)) return G4_ERR_UNSUPPORTED;
    return G4_OK;
  };

  EmbedArgs ea{d_tokens, d_idx, h->embed, h->ple_table, c.vocab, H, LP,
               (float)std::sqrt((double)H), (float)std::sqrt((double)P), h->x0, h->tok, h->err};
  set_tables(h, ea);
  {
    ProfScope ps(prof, "embed", (double)n * (H + LP) * 2);
    launch(embed_kernel, dim3(cdiv(H + LP, 8 * 256), n), dim3(256), 0, st, ea);
  }
  int pr_parts = 1;
  {
    StagedIn in;
    in.x = h->x0;
    in.x_stride = H;
    TRY(staged(h->pmp, in, h->sq_pr, LP, (long)kMaxNB * LP, &pr_parts, "gemv.ple_model_proj"));
  }
  {
    ProfScope ps(prof, "ple_combine", 0.0);
    launch(ple_combine_kernel, dim3(L, n), dim3(std::min(256, std::max(32, P))), 0, st, (const float*)h->sq_pr,
           pr_parts, (long)kMaxNB * LP, (const float*)h->tok, h->g_ppn, L, P, (float)(1.0 / std::sqrt((double)H)),
           (float)(1.0 / std::sqrt(2.0)), eps, h->ple);
  }
  float* cur = h->x0;
  auto next_x = [&]() { return cur == h->xb[0] ? h->xb[1] : h->xb[0]; };
  const int ts = h->trace_stride;
  int rple_parts = 1;
  for (int l = 0; l < L; ++l) {
    const Layer& Y = h->layers[l];
    const int nqd = c.num_q_heads * Y.d;
    int qkv_parts = 1, o_parts = 1, gu_parts = 1, d_parts = 1, pg_parts = 1;
    {  // QKV
      StagedIn in;
      in.x = cur;
      in.x_stride = H;
      in.g_a = Y.in_norm;
      if (l == 0) {
        in.pro = PRO_NORM;
      } else {
        const Layer& Pv = h->layers[l - 1];
        in.pro = PRO_RESID;
        in.r = h->sq_rple;
        in.r_stride = H;
        in.r_parts = rple_parts;
        in.r_part_stride = ps_h;
        in.g_r = Pv.post_ple_norm;
        in.lambda = Pv.lambda;
        in.x_out = next_x();
      }
      TRY(staged(Y.qkv, in, h->sq_qkv, h->sq_qkv_w, (long)kMaxNB * h->sq_qkv_w, &qkv_parts, "gemv.qkv", true));
      if (l > 0) {
        cur = in.x_out;
        if (h->trace)
          for (int i = 0; i < n; ++i)
            cudaMemcpyAsync(h->trace + ((size_t)((l - 1) * 2 + 1) * c.max_batch + i) * ts, cur + (size_t)i * H,
                            H * sizeof(float), cudaMemcpyDeviceToDevice, st);
      }
    }
    {
      ProfScope ps(prof, Y.full ? "attn.full" : "attn.sliding", 0.0);
      if (qkv_parts != 1) return G4_ERR_UNSUPPORTED;   // attention reads whole q, k, v rows
      launch_layer_attn(h, Y, h->sq_qkv, h->sq_qkv_w, n, d_slots, d_pos, Y.own != 0, st);
      if (h->trace)
        for (int i = 0; i < n; ++i)
          cudaMemcpyAsync(h->trace + ((size_t)(l * 2) * c.max_batch + i) * ts, h->attn + (size_t)i * nqd,
                          nqd * sizeof(float), cudaMemcpyDeviceToDevice, st);
    }
    {  // O
      StagedIn in;
      in.x = h->attn;
      in.x_stride = nqd;
      TRY(staged(Y.o, in, h->sq_rattn, H, ps_h, &o_parts, "gemv.o"));
    }
    {  // gate/up (raw rows: gate block j, up block j)
      StagedIn in;
      in.pro = PRO_RESID;
      in.x = cur;
      in.x_stride = H;
      in.r = h->sq_rattn;
      in.r_stride = H;
      in.r_parts = o_parts;
      in.r_part_stride = ps_h;
      in.g_r = Y.post_attn_norm;
      in.g_a = Y.pre_ffw_norm;
      in.x_out = next_x();
      TRY(staged(Y.gu, in, h->sq_gu, h->sq_gu_w, (long)kMaxNB * h->sq_gu_w, &gu_parts, "gemv.gate_up"));
      cur = in.x_out;
    }
    {  // down: input gelu(gate) * up
      StagedIn in;
      in.pro = PRO_GEGLU;
      in.x = h->sq_gu;
      in.x_stride = h->sq_gu_w;
      in.x_parts = gu_parts;
      in.x_part_stride = (long)kMaxNB * h->sq_gu_w;
      TRY(staged(Y.down, in, h->sq_rmlp, H, ps_h, &d_parts, "gemv.down"));
    }
    {  // per-layer-input gate (raw)
      StagedIn in;
      in.pro = PRO_RESID;
      in.x = cur;
      in.x_stride = H;
      in.r = h->sq_rmlp;
      in.r_stride = H;
      in.r_parts = d_parts;
      in.r_part_stride = ps_h;
      in.g_r = Y.post_ffw_norm;
      in.x_out = next_x();
      TRY(staged(Y.pg, in, h->sq_pg, P, (long)kMaxNB * P, &pg_parts, "gemv.ple_gate"));
      cur = in.x_out;
    }
    {  // per-layer projection: input gelu(gate) * ple_l
      StagedIn in;
      in.pro = PRO_PLEG;
      in.x = h->sq_pg;
      in.x_stride = P;
      in.x_parts = pg_parts;
      in.x_part_stride = (long)kMaxNB * P;
      in.ple = h->ple + (size_t)l * P;
      in.ple_stride = LP;
      TRY(staged(Y.pp, in, h->sq_rple, H, ps_h, &rple_parts, "gemv.ple_proj"));
    }
  }
  {  // final norm, lm_head, argmax (the branch comes in parts)
    const Layer& Pv = h->layers[L - 1];
    float* x_fin = next_x();
    bool done = false;
    if (lmhead_staged(h->lm.fmt)) {
      StagedIn in;
      in.pro = PRO_RESID;
      in.x = cur;
      in.x_stride = H;
      in.r = h->sq_rple;
      in.r_stride = H;
      in.r_parts = rple_parts;
      in.r_part_stride = ps_h;
      in.g_r = Pv.post_ple_norm;
      in.lambda = Pv.lambda;
      in.g_a = h->g_final;
      in.x_out = x_fin;
      ProfScope ps(prof, "gemv.lm_head_argmax", (double)h->lm.bytes);
      // the persistent GEMV's argmax counter (one past its row-group counters) is idle here
      unsigned* am_cnt = h->gemv_cnt + (size_t)(h->lm.n_rb / h->lm.R) * h->lm.ksplit;
      done = run_staged_argmax(h->lm, in, d_logits, c.vocab, d_next, n, eps, h->err, ctr(), h->am_val, h->am_idx,
                               am_cnt, h->sms, h->smem_optin, st);
    }
    GemvIO io;
    io.pro = PRO_RESID;
    io.x_in = cur;
    io.x_stride = H;
    io.norm_n = H;
    io.r_in = h->sq_rple;
    io.r_stride = H;
    io.r_parts = rple_parts;
    io.r_part_stride = ps_h;
    io.g_r = Pv.post_ple_norm;
    io.lambda = Pv.lambda;
    io.g_a = h->g_final;
    io.x_out = x_fin;
    io.logits = d_logits;
    io.logits_stride = c.vocab;
    io.next_ids = d_next;
    Scratch s{h->gemv_part, h->gemv_cnt, h->am_val, h->am_idx, h->err};
    if (!done) {
      ProfScope ps(prof, "gemv.lm_head_argmax", (double)h->lm.bytes);
      run_gemv(h->lm, EPI_ARGMAX, io, n, eps, s, h->sms, st, nullptr);
    }
    if (h->trace)
      for (int i = 0; i < n; ++i)
        cudaMemcpyAsync(h->trace + ((size_t)((L - 1) * 2 + 1) * c.max_batch + i) * ts, io.x_out + (size_t)i * H,
                        H * sizeof(float), cudaMemcpyDeviceToDevice, st);
  }
  CK(cudaGetLastError());
  return G4_OK;
}

g4_status run_step(g4_handle* h, cudaStream_t st, int n, const int* d_slots, const int* d_tokens, const int* d_idx,
                   const int* d_pos, int* d_next, float* d_logits, Prof* prof = nullptr, bool kv_first = false,
                   const int* keep_idx = nullptr, const int* keep_slots = nullptr, const int* keep_pos = nullptr,
                   int n_keep = -1) {
  if (h->mega_ok && h->mega_on && n <= 2 && !prof && !kv_first)
    return run_step_mega(h, st, n, d_slots, d_tokens, d_idx, d_pos, d_next, d_logits, false);
  if (gemv_staged_on() && n <= kMaxNB && !kv_first && n_keep < 0)
    return run_step_staged(h, st, n, d_slots, d_tokens, d_idx, d_pos, d_next, d_logits, prof);
  const g4_config& c = h->cfg;
  const int H = c.hidden, L = c.num_layers, P = c.ple_dim, LP = L * P;
  const float eps = c.rms_eps;
  Scratch s{h->gemv_part, h->gemv_cnt, h->am_val, h->am_idx, h->err};
  TcScratch tc{h->xt, h->tc_part, h->gemv_cnt, h->am_val, h->am_idx, h->err};

  EmbedArgs ea{d_tokens, d_idx, h->embed, h->ple_table, c.vocab, H, LP,
               (float)std::sqrt((double)H), (float)std::sqrt((double)P), h->x0, h->tok, h->err};
  set_tables(h, ea);
  {
    ProfScope ps(prof, "embed", (double)n * (H + LP) * 2);
    launch(embed_kernel, dim3(cdiv(H + LP, 8 * 256), n), dim3(256), 0, st, ea);
  }
  {
    ProfScope ps(prof, "gemv.ple_model_proj", (double)h->pmp.bytes);
    GemvIO io;
    io.pro = PRO_PLAIN;
    io.x_in = h->x0;
    io.x_stride = H;
    io.y = h->pr;
    io.y_stride = LP;
    run_gemv(h->pmp, EPI_STORE, io, n, eps, s, h->sms, st, &tc);
  }
  {
    ProfScope ps(prof, "ple_combine", 0.0);
    launch(ple_combine_kernel, dim3(L, n), dim3(std::min(256, std::max(32, P))), 0, st, (const float*)h->pr, 1, 0L,
           (const float*)h->tok, h->g_ppn, L, P, (float)(1.0 / std::sqrt((double)H)), (float)(1.0 / std::sqrt(2.0)),
           eps, h->ple);
  }

  float* cur = h->x0;
  auto next_x = [&]() { return cur == h->xb[0] ? h->xb[1] : h->xb[0]; };
  const int ts = h->trace_stride;
  const int l_tail = h->l_tail;
  const float* rple = h->r_ple;  // residual branch entering the next layer
  const float* ple_base = h->ple;
  for (int l = 0; l < L; ++l) {
    Layer& Y = h->layers[l];
    const int nqd = c.num_q_heads * Y.d;
    if (l == l_tail && l > 0 && n_keep >= 0 && n_keep < n) {
      if (n_keep == 0) return G4_OK;
      float* xg = next_x();
      launch(gather_rows_kernel, dim3(n_keep), dim3(256), 0, st, (const float*)cur, H, xg, H, keep_idx, H);
      launch(gather_rows_kernel, dim3(n_keep), dim3(256), 0, st, (const float*)h->r_ple, H, h->r_mlp, H, keep_idx, H);
      launch(gather_rows_kernel, dim3(n_keep), dim3(256), 0, st, ple_base, LP, h->pr, LP, keep_idx, LP);
      cur = xg;
      rple = h->r_mlp;
      ple_base = h->pr;
      d_slots = keep_slots;
      d_pos = keep_pos;
      n = n_keep;
    }
    {  // QKV
      GemvIO io;
      io.x_in = cur;
      io.x_stride = H;
      io.norm_n = H;
      io.g_a = Y.in_norm;
      if (l == 0) {
        io.pro = PRO_NORM;
      } else {
        const Layer& Pv = h->layers[l - 1];
        io.pro = PRO_RESID;
        io.r_in = rple;
        io.r_stride = H;
        io.g_r = Pv.post_ple_norm;
        io.lambda = Pv.lambda;
        io.x_out = next_x();
      }
      rple = h->r_ple;  // the gathered branch is used once
      io.y = h->qkv;
      io.y_stride = Y.qkv.n_valid;
      {
        ProfScope ps(prof, "gemv.qkv", (double)Y.qkv.bytes);
        run_gemv(Y.qkv, EPI_STORE, io, n, eps, s, h->sms, st, &tc);
      }
      if (l > 0) {
        cur = io.x_out;
        if (h->trace)
          for (int i = 0; i < n; ++i)
            cudaMemcpyAsync(h->trace + ((size_t)((l - 1) * 2 + 1) * c.max_batch + i) * ts, cur + (size_t)i * H,
                            H * sizeof(float), cudaMemcpyDeviceToDevice, st);
      }
    }
    {  // attention
      const Layer& Src = h->layers[Y.src];
      AttnArgs a{};
      a.qkv = h->qkv;
      a.qkv_stride = Y.qkv.n_valid;
      a.nq = c.num_q_heads;
      a.g_q = Y.q_norm;
      a.g_k = Y.k_norm;
      a.eps = eps;
      a.scale = Y.scale;
      a.window = Y.full ? 0 : c.sliding_window;
      a.own = Y.own && !kv_first;
      a.early = kv_first ? 0 : 1;  // prefill blocks: kv_write_kernel just wrote the rows
      kv_args(h, Src, a);
      a.t_max = c.max_context;
      a.max_batch = c.max_batch;
      a.rope_cos = h->cos_t[Y.full];
      a.rope_sin = h->sin_t[Y.full];
      a.slots = d_slots;
      a.positions = d_pos;
      a.out = h->attn;
      a.out_stride = nqd;
      const int hpc = attn_hpc(c.num_q_heads, n);
      const int max_keys = Y.full ? c.max_context : std::min(c.sliding_window, c.max_context);
      attn_plan(h->sms, c.num_q_heads, n, Y.d, max_keys, a);
      a.ws_ml = h->attn_ml;
      a.ws_o = h->attn_o;
      a.counters = h->attn_cnt;
      a.err = h->err;
      ProfScope ps(prof, Y.full ? "attn.full" : "attn.sliding", 0.0);
      if (kv_first && Y.own) launch_kv_write_any(a, Y.d, n, h->kv8, st);
      launch_attn_any(a, Y.d, hpc, n, h->kv8, mqa_on(c.num_q_heads, n), st);
      if (h->trace)
        for (int i = 0; i < n; ++i)
          cudaMemcpyAsync(h->trace + ((size_t)(l * 2) * c.max_batch + i) * ts, h->attn + (size_t)i * nqd,
                          nqd * sizeof(float), cudaMemcpyDeviceToDevice, st);
    }
    {  // O
      GemvIO io;
      io.pro = PRO_PLAIN;
      io.x_in = h->attn;
      io.x_stride = nqd;
      io.y = h->r_attn;
      io.y_stride = H;
      ProfScope ps(prof, "gemv.o", (double)Y.o.bytes);
      run_gemv(Y.o, EPI_STORE, io, n, eps, s, h->sms, st, &tc);
    }
    {  // gate/up
      GemvIO io;
      io.pro = PRO_RESID;
      io.x_in = cur;
      io.x_stride = H;
      io.norm_n = H;
      io.r_in = h->r_attn;
      io.r_stride = H;
      io.g_r = Y.post_attn_norm;
      io.lambda = 1.f;
      io.g_a = Y.pre_ffw_norm;
      io.x_out = next_x();
      io.y = h->act;
      io.y_stride = Y.F;
      {
        ProfScope ps(prof, "gemv.gate_up", (double)Y.gu.bytes);
        run_gemv(Y.gu, EPI_GEGLU, io, n, eps, s, h->sms, st, &tc);
      }
      cur = io.x_out;
    }
    {  // down
      GemvIO io;
      io.pro = PRO_PLAIN;
      io.x_in = h->act;
      io.x_stride = Y.F;
      io.y = h->r_mlp;
      io.y_stride = H;
      ProfScope ps(prof, "gemv.down", (double)Y.down.bytes);
      run_gemv(Y.down, EPI_STORE, io, n, eps, s, h->sms, st, &tc);
    }
    {  // PLE gate
      GemvIO io;
      io.pro = PRO_RESID;
      io.x_in = cur;
      io.x_stride = H;
      io.norm_n = H;
      io.r_in = h->r_mlp;
      io.r_stride = H;
      io.g_r = Y.post_ffw_norm;
      io.lambda = 1.f;
      io.g_a = nullptr;
      io.x_out = next_x();
      io.y = h->pg;
      io.y_stride = P;
      io.ple = ple_base + (size_t)l * P;
      io.ple_stride = LP;
      {
        ProfScope ps(prof, "gemv.ple_gate", (double)Y.pg.bytes);
        run_gemv(Y.pg, EPI_PLE, io, n, eps, s, h->sms, st, &tc);
      }
      cur = io.x_out;
    }
    {  // PLE proj
      GemvIO io;
      io.pro = PRO_PLAIN;
      io.x_in = h->pg;
      io.x_stride = P;
      io.y = h->r_ple;
      io.y_stride = H;
      ProfScope ps(prof, "gemv.ple_proj", (double)Y.pp.bytes);
      run_gemv(Y.pp, EPI_STORE, io, n, eps, s, h->sms, st, &tc);
    }
  }
  {  // final norm, lm_head, argmax
    const Layer& Pv = h->layers[L - 1];
    GemvIO io;
    io.pro = PRO_RESID;
    io.x_in = cur;
    io.x_stride = H;
    io.norm_n = H;
    io.r_in = h->r_ple;
    io.r_stride = H;
    io.g_r = Pv.post_ple_norm;
    io.lambda = Pv.lambda;
    io.g_a = h->g_final;
    io.x_out = next_x();
    io.logits = d_logits;
    io.logits_stride = c.vocab;
    io.next_ids = d_next;
    {
      ProfScope ps(prof, "gemv.lm_head_argmax", (double)h->lm.bytes);
      run_gemv(h->lm, EPI_ARGMAX, io, n, eps, s, h->sms, st, &tc);
    }
    if (h->trace)
      for (int i = 0; i < n; ++i)
        cudaMemcpyAsync(h->trace + ((size_t)((L - 1) * 2 + 1) * c.max_batch + i) * ts, io.x_out + (size_t)i * H,
                        H * sizeof(float), cudaMemcpyDeviceToDevice, st);
  }
  CK(cudaGetLastError());
  return G4_OK;
}

// ------------------------------------------------------------------- persistent step
// Units of one projection phase: K slices of spu supergroups, wpu warps per unit, upc units
// per CTA at a time.  Minimises rounds x supergroups per warp; ties go to fewer K slices.
// Persistent-step plan of a projection: K slices (at most max_ks, dividing the supergroups)
// that balance units of spu supergroups over the G CTAs; ring items of at most kItemMax bytes.
void mega_plan(const Lin& L, int G, int max_ks, MegaPhase& ph) {
  const int n_rg = L.n_rb / L.R;
  long best_cost = -1;
  for (int spu = L.S; spu >= 1; --spu) {
    if (L.S % spu) continue;
    const int ks = L.S / spu;
    if (ks > max_ks) continue;
    const long units = (long)n_rg * ks;
    const long cost = ((units + G - 1) / G) * spu;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      ph.spu = spu;
      ph.ksplit = ks;
      ph.n_units = (int)units;
    }
  }
  const size_t sgb = (size_t)L.R * (8 * kTileBytes + (L.fmt == G4_W4A16 ? kTileBytes : 0));
  ph.chunk_sg = (int)std::max<size_t>(1, std::min<size_t>(ph.spu, kItemMax / sgb));
}

void mega_lin(MegaPhase& ph, const Lin& L) {
  ph.qw = L.qw;
  ph.sc = L.sc;
  ph.fmt = L.fmt == G4_W4A16 ? FMT_W4A16 : FMT_BF16;
  ph.R = L.R;
  ph.n_rb = L.n_rb;
  ph.tiles = L.tiles;
  ph.S = L.S;
  ph.K = L.K;
  ph.n_valid = L.n_valid;
}

g4_status build_mega(g4_handle* h, cudaStream_t st) {
  const g4_config& c = h->cfg;
  const int H = c.hidden, L = c.num_layers, P = c.ple_dim, nq = c.num_q_heads;
  const int G = h->sms, NB = 2;
  if (H % 8 || h->kv8 || h->t4) return G4_OK;  // the persistent step: bf16 cache rows and tables only
  std::vector<MegaPhase> prog;
  size_t smem_f = 64;  // floats
  auto wred_f = [&]() { return (size_t)2 * kMegaWarps * 2 * NB * 32; };  // double-buffered warp partials
  auto note_full = [&](int K, int r_parts) { smem_f = std::max(smem_f, full_red(NB, K, r_parts) + 32 * NB + wred_f()); };
  auto note_slice = [&](const MegaPhase& ph) {
    const int sgk = ph.fmt == FMT_W4A16 ? 256 : 64;
    smem_f = std::max(smem_f, (size_t)NB * ph.spu * sgk + wred_f());
  };
  // K-slice partial buffers for the branches summed by the next residual update
  float *o_parts = nullptr, *d_parts = nullptr, *pmp_parts = nullptr;
  TRY(dalloc(h, &o_parts, (size_t)8 * NB * H));
  TRY(dalloc(h, &d_parts, (size_t)8 * NB * H));
  TRY(dalloc(h, &pmp_parts, (size_t)8 * NB * L * P));
  float* cur = h->x0;
  auto next_x = [&]() { return cur == h->xb[0] ? h->xb[1] : h->xb[0]; };
  {  // PMP: pr = W_pmp (E[t] sqrt H), K-slice partials
    MegaPhase ph{};
    ph.type = PH_PMP;
    mega_lin(ph, h->pmp);
    mega_plan(h->pmp, G, 8, ph);
    ph.in_mode = IN_EMBED;
    ph.x_stride = H;
    ph.y = pmp_parts;
    ph.y_stride = L * P;
    ph.y_part_stride = (long)NB * L * P;
    ph.epi = EPI_STORE;
    note_full(H, 0);
    prog.push_back(ph);
    MegaPhase pl{};
    pl.type = PH_PLE;
    pl.L = L;
    pl.P = P;
    pl.pr_parts = pmp_parts;
    pl.pr_nparts = ph.ksplit;
    pl.pr_part_stride = ph.y_part_stride;
    pl.g_ppn = h->g_ppn;
    pl.ple_table = h->ple_table;
    pl.ple_out = h->ple;
    pl.inv_sqrt_h = (float)(1.0 / std::sqrt((double)H));
    pl.inv_sqrt2 = (float)(1.0 / std::sqrt(2.0));
    pl.sqrt_p = (float)std::sqrt((double)P);
    smem_f = std::max(smem_f, (size_t)P + 64);
    prog.push_back(pl);
  }
  int prev_parts = 1;              // r_ple comes as one final vector
  for (int l = 0; l < L; ++l) {
    const Layer& Y = h->layers[l];
    const int nqd = nq * Y.d;
    {  // QKV (final rows: attention reads them)
      MegaPhase ph{};
      ph.type = PH_GEMV;
      mega_lin(ph, Y.qkv);
      mega_plan(Y.qkv, G, 1, ph);
      ph.x_stride = H;
      ph.g_a = Y.in_norm;
      if (l == 0) {
        ph.in_mode = IN_EMBED_NORM;
        ph.x_out = h->x0;
        note_full(H, 0);
      } else {
        const Layer& Pv = h->layers[l - 1];
        ph.in_mode = IN_RESID;
        ph.x_in = cur;
        ph.r_in = h->r_ple;
        ph.r_parts = prev_parts;
        ph.r_part_stride = 0;
        ph.r_stride = H;
        ph.g_r = Pv.post_ple_norm;
        ph.lambda = Pv.lambda;
        ph.x_out = next_x();
        cur = ph.x_out;
        note_full(H, prev_parts);
      }
      ph.y = h->qkv;
      ph.y_stride = Y.qkv.n_valid;
      ph.epi = EPI_STORE;
      prog.push_back(ph);
    }
    {  // attention
      const Layer& Src = h->layers[Y.src];
      MegaPhase ph{};
      ph.type = PH_ATTN;
      AttnArgs& a = ph.attn;
      a.qkv = h->qkv;
      a.qkv_stride = Y.qkv.n_valid;
      a.nq = nq;
      a.g_q = Y.q_norm;
      a.g_k = Y.k_norm;
      a.eps = c.rms_eps;
      a.scale = Y.scale;
      a.window = Y.full ? 0 : c.sliding_window;
      a.own = Y.own;
      kv_args(h, Src, a);
      a.t_max = c.max_context;
      a.max_batch = c.max_batch;
      a.rope_cos = h->cos_t[Y.full];
      a.rope_sin = h->sin_t[Y.full];
      a.out = h->attn;
      a.out_stride = nqd;
      const int max_keys = Y.full ? c.max_context : std::min(c.sliding_window, c.max_context);
      a.nsplit = attn_nsplit(h->sms, nq, 1, 1, max_keys);
      a.nstage = 1;
      a.ws_ml = h->attn_ml;
      a.ws_o = h->attn_o;
      a.counters = h->attn_cnt;
      a.err = h->err;
      ph.attn_d = Y.d;
      ph.attn_hpc = 1;
      ph.attn_units = NB * nq * a.nsplit;
      if ((size_t)NB * nq * a.nsplit * 2 > h->attn_ml_n || (size_t)NB * nq * a.nsplit * Y.d > h->attn_o_n)
        return G4_OK;  // workspace sized for another plan: keep the launch-per-phase path
      size_t ab = 0;
      switch (Y.d) {
        case 64: ab = attn_halves<64>() * attn_smem_bytes<64, 1>(1); break;
        case 128: ab = attn_halves<128>() * attn_smem_bytes<128, 1>(1); break;
        case 256: ab = attn_halves<256>() * attn_smem_bytes<256, 1>(1); break;
        default: ab = attn_halves<512>() * attn_smem_bytes<512, 1>(1); break;
      }
      smem_f = std::max(smem_f, (ab + 3) / 4);
      prog.push_back(ph);
    }
    {  // O: K-slice partials summed by the gate/up residual update
      MegaPhase ph{};
      ph.type = PH_GEMV;
      mega_lin(ph, Y.o);
      mega_plan(Y.o, G, 4, ph);
      ph.in_mode = IN_PLAIN;
      ph.x_in = h->attn;
      ph.x_stride = nqd;
      ph.y = o_parts;
      ph.y_stride = H;
      ph.y_part_stride = (long)NB * H;
      ph.epi = EPI_STORE;
      note_slice(ph);
      prog.push_back(ph);
      prev_parts = ph.ksplit;
    }
    {  // gate/up with GeGLU (final)
      MegaPhase ph{};
      ph.type = PH_GEMV;
      mega_lin(ph, Y.gu);
      mega_plan(Y.gu, G, 1, ph);
      ph.in_mode = IN_RESID;
      ph.x_in = cur;
      ph.x_stride = H;
      ph.r_in = o_parts;
      ph.r_parts = prev_parts;
      ph.r_part_stride = (long)NB * H;
      ph.r_stride = H;
      ph.g_r = Y.post_attn_norm;
      ph.lambda = 1.f;
      ph.g_a = Y.pre_ffw_norm;
      ph.x_out = next_x();
      cur = ph.x_out;
      ph.y = h->act;
      ph.y_stride = Y.F;
      ph.epi = EPI_GEGLU;
      note_full(H, prev_parts);
      prog.push_back(ph);
    }
    {  // down: partials
      MegaPhase ph{};
      ph.type = PH_GEMV;
      mega_lin(ph, Y.down);
      mega_plan(Y.down, G, 4, ph);
      ph.in_mode = IN_PLAIN;
      ph.x_in = h->act;
      ph.x_stride = Y.F;
      ph.y = d_parts;
      ph.y_stride = H;
      ph.y_part_stride = (long)NB * H;
      ph.epi = EPI_STORE;
      note_slice(ph);
      prog.push_back(ph);
      prev_parts = ph.ksplit;
    }
    {  // PLE gate (final, gelu * ple_l)
      MegaPhase ph{};
      ph.type = PH_GEMV;
      mega_lin(ph, Y.pg);
      mega_plan(Y.pg, G, 1, ph);
      ph.in_mode = IN_RESID;
      ph.x_in = cur;
      ph.x_stride = H;
      ph.r_in = d_parts;
      ph.r_parts = prev_parts;
      ph.r_part_stride = (long)NB * H;
      ph.r_stride = H;
      ph.g_r = Y.post_ffw_norm;
      ph.lambda = 1.f;
      ph.g_a = nullptr;
      ph.x_out = next_x();
      cur = ph.x_out;
      ph.y = h->pg;
      ph.y_stride = P;
      ph.epi = EPI_PLE;
      ph.ple = h->ple + (size_t)l * P;
      ph.ple_stride = L * P;
      note_full(H, prev_parts);
      prog.push_back(ph);
    }
    {  // PLE proj (final r_ple)
      MegaPhase ph{};
      ph.type = PH_GEMV;
      mega_lin(ph, Y.pp);
      mega_plan(Y.pp, G, 1, ph);
      ph.in_mode = IN_PLAIN;
      ph.x_in = h->pg;
      ph.x_stride = P;
      ph.y = h->r_ple;
      ph.y_stride = H;
      ph.epi = EPI_STORE;
      note_slice(ph);
      prog.push_back(ph);
      prev_parts = 1;
    }
  }
  {  // lm_head + argmax
    const Layer& Pv = h->layers[L - 1];
    MegaPhase ph{};
    ph.type = PH_LMHEAD;
    mega_lin(ph, h->lm);
    mega_plan(h->lm, G, 1, ph);
    ph.epi = EPI_ARGMAX;
    ph.in_mode = IN_RESID;
    ph.x_in = cur;
    ph.x_stride = H;
    ph.r_in = h->r_ple;
    ph.r_parts = 1;
    ph.r_stride = H;
    ph.g_r = Pv.post_ple_norm;
    ph.lambda = Pv.lambda;
    ph.g_a = h->g_final;
    ph.x_out = next_x();
    note_full(H, 1);
    prog.push_back(ph);
    MegaPhase am{};
    am.type = PH_ARGMAX;
    prog.push_back(am);
  }
  {
    static const char* kLayerNames[] = {"mega.qkv", "mega.attn", "mega.o", "mega.gate_up", "mega.down",
                                        "mega.ple_gate", "mega.ple_proj"};
    h->mega_names.clear();
    h->mega_names.push_back("mega.ple_model_proj");
    h->mega_names.push_back("mega.ple_combine");
    for (int l = 0; l < L; ++l)
      for (const char* nm : kLayerNames) h->mega_names.push_back(nm);
    h->mega_names.push_back("mega.lm_head");
    h->mega_names.push_back("mega.argmax");
  }
  // per-layer trace points: residual after layer l is materialised by layer l+1's QKV phase
  // (the lm_head phase for the last layer); attention output of layer l is read by its O phase
  {
    for (MegaPhase& ph : prog) {
      ph.trace_x = -1;
      ph.trace_attn = -1;
    }
    int idx = 2;
    for (int l = 0; l < L; ++l) {
      if (l > 0) prog[idx].trace_x = l - 1;      // QKV of layer l
      prog[idx + 2].trace_attn = l;               // O of layer l
      prog[idx + 2].trace_attn_width = nq * h->layers[l].d;
      idx += 7;
    }
    prog[idx].trace_x = L - 1;                    // lm_head
  }
  h->mega_smem = kRingBytes + smem_f * 4;
  int optin = init_kernel_attrs(h->device);
  if ((int)h->mega_smem > optin) return G4_OK;
  int nb1 = 0, nb2 = 0;
  CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb1, mega_step_kernel<1>, kMegaThreads, h->mega_smem));
  CK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb2, mega_step_kernel<2>, kMegaThreads, h->mega_smem));
  if (nb1 < 1 || nb2 < 1) return G4_OK;
  h->mega_grid = G;
  h->mega_n = (int)prog.size();
  TRY(dalloc(h, &h->mega_stamps, prog.size() + 1));
  TRY(dalloc(h, &h->mega_phases, prog.size()));
  CK(cudaMemcpyAsync(h->mega_phases, prog.data(), prog.size() * sizeof(MegaPhase), cudaMemcpyHostToDevice, st));
  TRY(dalloc(h, &h->mega_bar, 2));
  TRY(dalloc(h, &h->mega_am_val, (size_t)NB * G));
  TRY(dalloc(h, &h->mega_am_idx, (size_t)NB * G));
  CK(cudaStreamSynchronize(st));
  h->mega_ok = true;
  return G4_OK;
}

g4_status run_step_mega(g4_handle* h, cudaStream_t st, int n, const int* d_slots, const int* d_tokens,
                        const int* d_idx, const int* d_pos, int* d_next, float* d_logits, bool stamps) {
  MegaArgs a{};
  a.stamps = stamps ? h->mega_stamps : nullptr;
  a.phases = h->mega_phases;
  a.n_phases = h->mega_n;
  a.nb = n;
  a.slots = d_slots;
  a.positions = d_pos;
  a.tokens = d_tokens;
  a.tok_idx = d_idx;
  a.embed = h->embed;
  a.H = h->cfg.hidden;
  a.V = h->cfg.vocab;
  a.sqrt_h = (float)std::sqrt((double)h->cfg.hidden);
  a.eps = h->cfg.rms_eps;
  a.barrier = h->mega_bar;
  a.am_val = h->mega_am_val;
  a.am_idx = h->mega_am_idx;
  a.next_ids = d_next;
  a.logits = d_logits;
  a.logits_stride = h->cfg.vocab;
  a.err = h->err;
  a.trace = h->trace;
  a.trace_stride = h->trace_stride;
  a.max_batch = h->cfg.max_batch;
  CK(cudaMemsetAsync(h->mega_bar, 0, 2 * sizeof(unsigned), st));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h->mega_grid);
  cfg.blockDim = dim3(kMegaThreads);
  cfg.dynamicSmemBytes = h->mega_smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (n == 1) CK(cudaLaunchKernelEx(&cfg, mega_step_kernel<1>, a));
  else CK(cudaLaunchKernelEx(&cfg, mega_step_kernel<2>, a));
  return G4_OK;
}

bool is_pow2_dim(int d) { return d == 64 || d == 128 || d == 256 || d == 512; }

// Pages for positions [0, n) of `slot` (paged cache): take the missing ones from the pool and
// upload the slot's page-table row.
g4_status kv_reserve_impl(g4_handle* h, cudaStream_t st, int slot, int n) {
  const int need = cdiv(n, 1 << h->page_shift);
  int& have = h->slot_pages[slot];
  if (need <= have) return G4_OK;
  if (need - have > (int)h->free_pages.size()) return G4_ERR_OOM;
  int* row = h->pt_host.data() + (size_t)slot * h->max_pages;
  const int first = have;
  for (; have < need; ++have) {
    row[have] = h->free_pages.back();
    h->free_pages.pop_back();
  }
  CK(cudaMemcpyAsync(h->page_table + (size_t)slot * h->max_pages + first, row + first, (need - first) * sizeof(int),
                     cudaMemcpyHostToDevice, st));
  return G4_OK;
}

g4_status validate(const g4_config* c) {
  if (!c) return G4_ERR_INVALID_ARG;
  if (c->num_layers < 1 || c->num_kv_shared_layers < 0 || c->num_kv_shared_layers >= c->num_layers)
    return G4_ERR_INVALID_ARG;
  if (c->hidden < 32 || c->num_q_heads < 1 || c->vocab < 1 || c->ple_dim < 1 || c->mlp < 32 || c->mlp_shared < 32)
    return G4_ERR_INVALID_ARG;
  if (c->max_batch < 1 || c->max_context < 1 || c->full_every < 1 || c->sliding_window < 1) return G4_ERR_INVALID_ARG;
  if (c->weight_format != G4_BF16 && c->weight_format != G4_W4A16) return G4_ERR_INVALID_ARG;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta_sliding > 0.f) || !(c->rope_theta_full > 0.f)) return G4_ERR_INVALID_ARG;
  if (c->num_kv_heads != 1 || c->group_size != 32) return G4_ERR_UNSUPPORTED;
  if (!is_pow2_dim(c->head_dim_sliding) || !is_pow2_dim(c->head_dim_full)) return G4_ERR_UNSUPPORTED;
  if (c->hidden % 32 || c->mlp % 32 || c->mlp_shared % 32 || c->ple_dim % 32) return G4_ERR_UNSUPPORTED;
  if (c->max_batch > 64 || c->ple_dim > 1024 || c->hidden > 8192) return G4_ERR_UNSUPPORTED;
  if (c->kv_format != G4_KV_BF16 && c->kv_format != G4_KV_INT8) return G4_ERR_INVALID_ARG;
  if (c->kv_page_size < 0 || c->kv_pages < 0) return G4_ERR_INVALID_ARG;
  if (c->kv_page_size > 0 && (c->kv_page_size < 16 || (c->kv_page_size & (c->kv_page_size - 1))))
    return G4_ERR_UNSUPPORTED;  // pages of a power of two >= 16 positions
  if (c->table_format != G4_BF16 && c->table_format != G4_W4A16) return G4_ERR_INVALID_ARG;
  return G4_OK;
}

g4_status create_impl(g4_handle* h, const g4_config* cfg, const g4_weights* w, cudaStream_t st) {
  const g4_config& c = *cfg;
  const int L = c.num_layers, H = c.hidden, P = c.ple_dim, nq = c.num_q_heads;
  const int first = L - c.num_kv_shared_layers;
  const int fmt = c.weight_format;
  std::vector<RbSrc> keep;
  h->embed = static_cast<const __nv_bfloat16*>(w->embed);
  h->ple_table = static_cast<const __nv_bfloat16*>(w->ple_table);
  h->g_ppn = static_cast<const __nv_bfloat16*>(w->ple_proj_norm);
  h->g_final = static_cast<const __nv_bfloat16*>(w->final_norm);
  if (!h->embed || !h->ple_table || !h->g_ppn || !h->g_final || !w->layers || !w->ple_model_proj.w)
    return G4_ERR_INVALID_ARG;
  if (fmt == G4_W4A16 && !w->ple_model_proj.scales) return G4_ERR_INVALID_ARG;
  if (c.table_format == G4_W4A16) {
    if (!w->embed_scales || !w->ple_table_scales) return G4_ERR_INVALID_ARG;
    h->t4 = true;
    h->embed_q = static_cast<const uint32_t*>(w->embed);
    h->embed_s = static_cast<const __nv_bfloat16*>(w->embed_scales);
    h->ple_q = static_cast<const uint32_t*>(w->ple_table);
    h->ple_s = static_cast<const __nv_bfloat16*>(w->ple_table_scales);
  }

  // layer schedule: type, share source, ownership ("One TPU chip, eight agents", The engine)
  std::vector<int> full(L), src(L);
  int last_of[2] = {-1, -1};
  for (int l = 0; l < L; ++l) full[l] = (l % c.full_every) == c.full_every - 1;
  for (int l = 0; l < first; ++l) last_of[full[l]] = l;
  for (int l = 0; l < L; ++l) src[l] = (l < first || last_of[full[l]] < 0) ? l : last_of[full[l]];

  h->layers.resize(L);
  int n_own = 0;
  for (int l = 0; l < L; ++l) {
    Layer& Y = h->layers[l];
    const g4_layer_weights& lw = w->layers[l];
    Y.full = full[l];
    Y.d = Y.full ? c.head_dim_full : c.head_dim_sliding;
    Y.F = l >= first ? c.mlp_shared : c.mlp;
    Y.src = src[l];
    Y.own = src[l] == l;
    Y.kv = Y.own ? n_own++ : -1;
    const float sc = Y.full ? c.attn_scale_full : c.attn_scale_sliding;
    Y.scale = sc != 0.f ? sc : (float)(1.0 / std::sqrt((double)Y.d));
    Y.lambda = lw.layer_scale;
    Y.in_norm = (const __nv_bfloat16*)lw.in_norm;
    Y.post_attn_norm = (const __nv_bfloat16*)lw.post_attn_norm;
    Y.pre_ffw_norm = (const __nv_bfloat16*)lw.pre_ffw_norm;
    Y.post_ffw_norm = (const __nv_bfloat16*)lw.post_ffw_norm;
    Y.post_ple_norm = (const __nv_bfloat16*)lw.post_ple_norm;
    Y.q_norm = (const __nv_bfloat16*)lw.q_norm;
    Y.k_norm = (const __nv_bfloat16*)lw.k_norm;
    if (!Y.in_norm || !Y.post_attn_norm || !Y.pre_ffw_norm || !Y.post_ffw_norm || !Y.post_ple_norm || !Y.q_norm)
      return G4_ERR_INVALID_ARG;
    const g4_linear* need[] = {&lw.q, &lw.o, &lw.gate, &lw.up, &lw.down, &lw.ple_gate, &lw.ple_proj};
    for (const g4_linear* p : need)
      if (!p->w || (fmt == G4_W4A16 && !p->scales)) return G4_ERR_INVALID_ARG;
    if (Y.own && (!lw.k.w || !lw.v.w || !Y.k_norm || (fmt == G4_W4A16 && (!lw.k.scales || !lw.v.scales))))
      return G4_ERR_INVALID_ARG;
    const int nqd = nq * Y.d;
    std::vector<Seg> qkv = {{lw.q.w, lw.q.scales, nqd}};
    if (Y.own) {
      qkv.push_back({lw.k.w, lw.k.scales, Y.d});
      qkv.push_back({lw.v.w, lw.v.scales, Y.d});
    }
    TRY(build_lin(h, fmt, H, qkv, false, &Y.qkv, st, keep));
    TRY(build_lin(h, fmt, nqd, {{lw.o.w, lw.o.scales, H}}, false, &Y.o, st, keep));
    TRY(build_lin(h, fmt, H, {{lw.gate.w, lw.gate.scales, Y.F}, {lw.up.w, lw.up.scales, Y.F}}, true, &Y.gu, st, keep));
    TRY(build_lin(h, fmt, Y.F, {{lw.down.w, lw.down.scales, H}}, false, &Y.down, st, keep));
    TRY(build_lin(h, fmt, H, {{lw.ple_gate.w, lw.ple_gate.scales, P}}, false, &Y.pg, st, keep));
    TRY(build_lin(h, fmt, P, {{lw.ple_proj.w, lw.ple_proj.scales, H}}, false, &Y.pp, st, keep));
    for (Lin* Ln : {&Y.qkv, &Y.o, &Y.gu, &Y.down, &Y.pg, &Y.pp}) plan_lin(*Ln, h->sms, false);
  }
  TRY(build_lin(h, fmt, H, {{w->ple_model_proj.w, w->ple_model_proj.scales, L * P}}, false, &h->pmp, st, keep));
  plan_lin(h->pmp, h->sms, false);
  if (h->t4)
    TRY(build_lin(h, G4_W4A16, H, {{w->embed, w->embed_scales, c.vocab}}, false, &h->lm, st, keep));
  else
    TRY(build_lin(h, G4_BF16, H, {{w->embed, nullptr, c.vocab}}, false, &h->lm, st, keep));
  plan_lin(h->lm, h->sms, true);

  // KV cache: owning layers only.  Static: [max_batch][max_context] rows of d values for K
  // and for V.  Paged: a pool of n_pages pages of page_size rows, and one page table.
  h->kv8 = c.kv_format == G4_KV_INT8;
  size_t kv_rows = (size_t)c.max_batch * c.max_context;
  if (c.kv_page_size > 0) {
    while ((1 << h->page_shift) < c.kv_page_size) ++h->page_shift;
    h->max_pages = cdiv(c.max_context, c.kv_page_size);
    h->n_pages = c.kv_pages > 0 ? c.kv_pages : c.max_batch * h->max_pages;
    kv_rows = (size_t)h->n_pages << h->page_shift;
    h->pt_host.assign((size_t)c.max_batch * h->max_pages, -1);
    h->slot_pages.assign(c.max_batch, 0);
    for (int pg = h->n_pages - 1; pg >= 0; --pg) h->free_pages.push_back(pg);  // page 0 taken first
    TRY(dalloc(h, &h->page_table, h->pt_host.size()));
    CK(cudaMemcpyAsync(h->page_table, h->pt_host.data(), h->pt_host.size() * sizeof(int), cudaMemcpyHostToDevice, st));
    CK(cudaStreamSynchronize(st));
  }
  h->kc.resize(n_own);
  h->vc.resize(n_own);
  h->ksc.assign(n_own, nullptr);
  h->vsc.assign(n_own, nullptr);
  for (int l = 0; l < L; ++l) {
    const Layer& Y = h->layers[l];
    if (!Y.own) continue;
    const size_t nb = kv_rows * Y.d * (h->kv8 ? 1 : 2);
    uint8_t *kb = nullptr, *vb = nullptr;
    TRY(dalloc(h, &kb, nb));
    TRY(dalloc(h, &vb, nb));
    CK(cudaMemsetAsync(kb, 0, nb, st));
    CK(cudaMemsetAsync(vb, 0, nb, st));
    h->kc[Y.kv] = kb;
    h->vc[Y.kv] = vb;
    if (h->kv8) {
      TRY(dalloc(h, &h->ksc[Y.kv], kv_rows));
      TRY(dalloc(h, &h->vsc[Y.kv], kv_rows));
      CK(cudaMemsetAsync(h->ksc[Y.kv], 0, kv_rows * 4, st));
      CK(cudaMemsetAsync(h->vsc[Y.kv], 0, kv_rows * 4, st));
    }
  }
  // RoPE tables (fp64 angles, rounded to fp32)
  for (int t = 0; t < 2; ++t) {
    const int d = t ? c.head_dim_full : c.head_dim_sliding;
    const double theta = t ? c.rope_theta_full : c.rope_theta_sliding;
    std::vector<float> cs((size_t)c.max_context * d / 2), sn(cs.size());
    for (int i = 0; i < d / 2; ++i) {
      const double inv = std::pow(theta, -2.0 * i / d);
      for (int p = 0; p < c.max_context; ++p) {
        const double ang = (double)p * inv;
        cs[(size_t)p * (d / 2) + i] = (float)std::cos(ang);
        sn[(size_t)p * (d / 2) + i] = (float)std::sin(ang);
      }
    }
    TRY(dalloc(h, &h->cos_t[t], cs.size()));
    TRY(dalloc(h, &h->sin_t[t], sn.size()));
    CK(cudaMemcpy(h->cos_t[t], cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(h->sin_t[t], sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
  }
  h->l_tail = L;
  while (h->l_tail > 0 && !h->layers[h->l_tail - 1].own) --h->l_tail;
  // activations: rows for a step of max_batch sequences or a prefill block of kPrefillRows
  // tokens (rows of one sequence at consecutive positions)
  const int B = std::max(c.max_batch, kPrefillRows);
  h->rows = B;
  const int dmax = std::max(c.head_dim_full, c.head_dim_sliding);
  const int Fmax = std::max(c.mlp, c.mlp_shared);
  TRY(dalloc(h, &h->x0, (size_t)B * H));
  TRY(dalloc(h, &h->xb[0], (size_t)B * H));
  TRY(dalloc(h, &h->xb[1], (size_t)B * H));
  TRY(dalloc(h, &h->tok, (size_t)B * L * P));
  TRY(dalloc(h, &h->pr, (size_t)B * L * P));
  TRY(dalloc(h, &h->ple, (size_t)B * L * P));
  TRY(dalloc(h, &h->qkv, (size_t)B * (nq + 2) * dmax));
  TRY(dalloc(h, &h->attn, (size_t)B * nq * dmax));
  TRY(dalloc(h, &h->r_attn, (size_t)B * H));
  TRY(dalloc(h, &h->act, (size_t)B * Fmax));
  TRY(dalloc(h, &h->r_mlp, (size_t)B * H));
  TRY(dalloc(h, &h->pg, (size_t)B * P));
  TRY(dalloc(h, &h->r_ple, (size_t)B * H));
  {  // staged decode step buffers: kSgMaxParts parts of kMaxNB rows
    h->sq_qkv_w = (nq + 2) * dmax;
    h->sq_gu_w = 2 * Fmax;
    const size_t R4 = (size_t)kSgMaxParts * kMaxNB;
    TRY(dalloc(h, &h->sq_qkv, R4 * h->sq_qkv_w));
    TRY(dalloc(h, &h->sq_rattn, R4 * H));
    TRY(dalloc(h, &h->sq_gu, R4 * h->sq_gu_w));
    TRY(dalloc(h, &h->sq_rmlp, R4 * H));
    TRY(dalloc(h, &h->sq_pg, R4 * P));
    TRY(dalloc(h, &h->sq_rple, R4 * H));
    TRY(dalloc(h, &h->sq_pr, R4 * L * P));
    const size_t nctr = (size_t)kSgCtrSlots * 2 * kSgMaxParts;
    TRY(dalloc(h, &h->sg_ctr, nctr));
    CK(cudaMemsetAsync(h->sg_ctr, 0, nctr * sizeof(unsigned), st));
  }
  // GEMV scratch: partials of the widest split, one counter per row group (+1 for argmax)
  size_t part = 1, cnt = 1;
  auto acc_lin = [&](const Lin& Ln) {
    part = std::max(part, (size_t)Ln.ksplit * kMaxNB * Ln.n_rb * 32);
    cnt = std::max(cnt, (size_t)(Ln.n_rb / Ln.R) * Ln.ksplit + 1);
  };
  for (const Layer& Y : h->layers)
    for (const Lin* Ln : {&Y.qkv, &Y.o, &Y.gu, &Y.down, &Y.pg, &Y.pp}) acc_lin(*Ln);
  acc_lin(h->pmp);
  acc_lin(h->lm);
  // tensor-core GEMM scratch: activation tiles for the widest K, split-K partials
  size_t xtb = 16, tcp = 1;
  auto acc_tc = [&](const Lin& Ln, bool whole) {
    int ks, kbps;
    tc_plan(Ln, h->sms, whole, &ks, &kbps);
    xtb = std::max(xtb, (size_t)tc_nkb(Ln) * 2 * 64 * 128);
    tcp = std::max(tcp, (size_t)ks * 64 * (Ln.n_rb / 4) * 128);
    cnt = std::max(cnt, (size_t)(Ln.n_rb / 4) + 1);
  };
  for (const Layer& Y : h->layers)
    for (const Lin* Ln : {&Y.qkv, &Y.o, &Y.gu, &Y.down, &Y.pg, &Y.pp}) acc_tc(*Ln, false);
  acc_tc(h->pmp, false);
  acc_tc(h->lm, true);
  h->xt_bytes = xtb;
  h->tc_part_floats = tcp;
  TRY(dalloc(h, &h->xt, xtb));
  CK(cudaMemsetAsync(h->xt, 0, xtb, st));
  TRY(dalloc(h, &h->tc_part, tcp));
  h->gemv_part_floats = part;
  h->gemv_cnt_n = cnt;
  TRY(dalloc(h, &h->gemv_part, part));
  TRY(dalloc(h, &h->gemv_cnt, cnt));
  CK(cudaMemsetAsync(h->gemv_cnt, 0, cnt * sizeof(unsigned), st));
  h->am_n = std::max((size_t)kMaxNB * (h->lm.n_rb / h->lm.R) * h->lm.ksplit, (size_t)64 * (h->lm.n_rb / 4));
  TRY(dalloc(h, &h->am_val, h->am_n));
  TRY(dalloc(h, &h->am_idx, h->am_n));
  // attention scratch for the largest (nb * nsplit) over batch sizes
  size_t ml = 1, ao = 1;
  for (int nb = 1; nb <= std::max(B, 2); ++nb) {  // the persistent step plans for 2 rows
    const int hpc = attn_hpc(nq, nb);
    for (int t = 0; t < 2; ++t) {
      const int d = t ? c.head_dim_full : c.head_dim_sliding;
      const int keys = t ? c.max_context : std::min(c.sliding_window, c.max_context);
      const int ns = attn_nsplit(h->sms, nq, hpc, nb, keys);
      const int ns1 = attn_nsplit(h->sms, nq, 1, 1, keys);  // persistent step: nb=1 plan, 2 rows
      const int nsm = mqa_nsplit(h->sms, nb, keys);
      ml = std::max({ml, (size_t)nb * nq * ns * 2, (size_t)2 * nq * ns1 * 2, (size_t)nb * nq * nsm * 2});
      ao = std::max({ao, (size_t)nb * nq * ns * d, (size_t)2 * nq * ns1 * d, (size_t)nb * nq * nsm * d});
    }
  }
  h->attn_ml_n = ml;
  h->attn_o_n = ao;
  TRY(dalloc(h, &h->attn_ml, ml));
  TRY(dalloc(h, &h->attn_o, ao));
  TRY(dalloc(h, &h->attn_cnt, (size_t)std::max(B, 2) * nq));
  CK(cudaMemsetAsync(h->attn_cnt, 0, (size_t)std::max(B, 2) * nq * sizeof(unsigned), st));
  TRY(dalloc(h, &h->err, 1));
  CK(cudaMemsetAsync(h->err, 0, sizeof(int), st));
  TRY(dalloc(h, &h->step_next, B));
  TRY(dalloc(h, &h->step_logits, (size_t)B * c.vocab));  // only the rows that end a sequence are read
  CK(cudaStreamSynchronize(st));
  TRY(build_mega(h, st));
  return G4_OK;
}

void destroy(g4_handle* h) {
  DeviceGuard dg(h->device);
  cudaDeviceSynchronize();
  for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
  for (void* p : h->allocs) cudaFree(p);
  if (h->pf_buf) cudaFree(h->pf_buf);
  delete h;
}

}  // namespace

// =================================================================================== C ABI
extern "C" {

const char* g4_status_string(g4_status s) {
  switch (s) {
    case G4_OK: return "ok";
    case G4_ERR_INVALID_ARG: return "invalid argument";
    case G4_ERR_UNSUPPORTED: return "unsupported configuration";
    case G4_ERR_OOM: return "out of device memory";
    case G4_ERR_CUDA: return "CUDA error";
    case G4_ERR_CONTEXT_OVERFLOW: return "context overflow";
    case G4_ERR_TIMEOUT: return "device wait timed out";
    case G4_ERR_DEVICE_CHECK: return "device-side argument check failed";
  }
  return "unknown status";
}

const char* g4_last_cuda_error(void) { return g_last_cuda.c_str(); }

g4_status g4_create(const g4_config* cfg, const g4_weights* weights, int device, g4_handle** out) {
  if (!out) return G4_ERR_INVALID_ARG;
  *out = nullptr;
  g4_status v = validate(cfg);
  if (v != G4_OK) return v;
  if (!weights) return G4_ERR_INVALID_ARG;
  DEVICE_GUARD(device);
  const int optin = init_kernel_attrs(device);
  g4_handle* h = new g4_handle();
  h->cfg = *cfg;
  h->device = device;
  h->smem_optin = optin;
  if (const char* fa = getenv("G4_FAIL_ALLOC_AT")) h->fail_at = atoi(fa);
  cudaError_t e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, device);
  if (!cuda_ok(e, "cudaDeviceGetAttribute")) { delete h; return G4_ERR_CUDA; }
  cudaStream_t st = nullptr;
  e = cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking);
  if (!cuda_ok(e, "cudaStreamCreate")) { delete h; return G4_ERR_CUDA; }
  g4_status s = create_impl(h, cfg, weights, st);
  cudaStreamSynchronize(st);
  cudaStreamDestroy(st);
  if (s != G4_OK) { destroy(h); return s; }
  h->fail_at = 0;  // the hook covers g4_create only
  *out = h;
  return G4_OK;
}

void g4_free(g4_handle* h) {
  if (h) destroy(h);
}

int64_t g4_device_bytes(const g4_handle* h) { return h ? (int64_t)h->bytes : 0; }

g4_status g4_kv_reserve(g4_handle* h, g4_stream stream, int32_t slot, int32_t n_positions) {
  if (!h || slot < 0 || slot >= h->cfg.max_batch || n_positions < 0) return G4_ERR_INVALID_ARG;
  if (n_positions > h->cfg.max_context) return G4_ERR_CONTEXT_OVERFLOW;
  if (!h->page_table) return G4_OK;
  DEVICE_GUARD(h->device);
  return kv_reserve_impl(h, reinterpret_cast<cudaStream_t>(stream), slot, n_positions);
}

g4_status g4_kv_release(g4_handle* h, g4_stream stream, int32_t slot) {
  if (!h || slot < 0 || slot >= h->cfg.max_batch) return G4_ERR_INVALID_ARG;
  if (!h->page_table) return G4_OK;
  DEVICE_GUARD(h->device);
  int& have = h->slot_pages[slot];
  if (have == 0) return G4_OK;
  int* row = h->pt_host.data() + (size_t)slot * h->max_pages;
  for (int k = have - 1; k >= 0; --k) {
    h->free_pages.push_back(row[k]);
    row[k] = -1;
  }
  CK(cudaMemcpyAsync(h->page_table + (size_t)slot * h->max_pages, row, have * sizeof(int), cudaMemcpyHostToDevice,
                     reinterpret_cast<cudaStream_t>(stream)));
  have = 0;
  return G4_OK;
}

int32_t g4_kv_pages_free(const g4_handle* h) {
  if (!h || !h->page_table) return -1;
  return (int32_t)h->free_pages.size();
}

int32_t g4_step_mode(const g4_handle* h, int32_t n_seq) {
  if (!h) return -1;
  return (h->mega_ok && h->mega_on && n_seq <= 2) ? 1 : 0;
}

g4_status g4_set_step_mode(g4_handle* h, int32_t mode) {
  if (!h || (mode != 0 && mode != 1)) return G4_ERR_INVALID_ARG;
  if (mode == 1 && !h->mega_ok) return G4_ERR_UNSUPPORTED;
  h->mega_on = mode == 1;
  return G4_OK;
}

g4_status g4_set_trace(g4_handle* h, float* d_trace, int64_t capacity_floats) {
  if (!h) return G4_ERR_INVALID_ARG;
  const g4_config& c = h->cfg;
  const int stride = std::max(c.hidden, c.num_q_heads * std::max(c.head_dim_full, c.head_dim_sliding));
  if (d_trace && capacity_floats < (int64_t)c.num_layers * 2 * c.max_batch * stride) return G4_ERR_INVALID_ARG;
  h->trace = d_trace;
  h->trace_stride = stride;
  return G4_OK;
}

g4_status g4_decode_step(g4_handle* h, g4_stream stream, int32_t n_seq, const int32_t* d_slots,
                         const int32_t* d_tokens, const int32_t* d_positions, int32_t* d_next_ids, float* d_logits) {
  if (!h || !d_slots || !d_tokens || !d_positions || !d_next_ids) return G4_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > h->cfg.max_batch) return G4_ERR_INVALID_ARG;
  DEVICE_GUARD(h->device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (st == nullptr) {  // the legacy default stream cannot be captured: launch directly
    return run_step(h, st, n_seq, d_slots, d_tokens, nullptr, d_positions, d_next_ids, d_logits);
  }
  GraphKey key{n_seq, g4_step_mode(h, n_seq), d_slots, d_tokens, d_positions, d_next_ids, d_logits, h->trace};
  auto it = h->graphs.find(key);
  if (it == h->graphs.end()) {
    if (h->graphs.size() >= 16) {
      for (auto& kv : h->graphs) cudaGraphExecDestroy(kv.second);
      h->graphs.clear();
    }
    CK(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
    g4_status s = run_step(h, st, n_seq, d_slots, d_tokens, nullptr, d_positions, d_next_ids, d_logits);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(st, &g);
    if (s != G4_OK) { if (g) cudaGraphDestroy(g); return s; }
    CK(e);
    cudaGraphExec_t ex = nullptr;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    CK(e);
    it = h->graphs.emplace(key, ex).first;
  }
  CK(cudaGraphLaunch(it->second, st));
  return G4_OK;
}

g4_status g4_prefill(g4_handle* h, g4_stream stream, int32_t n_seq, const int32_t* slots, const int32_t* offsets,
                     const int32_t* start_pos, const int32_t* d_tokens, int32_t* d_next_ids, float* d_logits) {
  if (!h || !slots || !offsets || !start_pos || !d_tokens || !d_next_ids) return G4_ERR_INVALID_ARG;
  const g4_config& c = h->cfg;
  if (n_seq < 1 || n_seq > c.max_batch) return G4_ERR_INVALID_ARG;
  std::vector<int> len(n_seq), order(n_seq);
  std::vector<char> used(c.max_batch, 0);
  for (int i = 0; i < n_seq; ++i) {
    len[i] = offsets[i + 1] - offsets[i];
    if (len[i] < 1 || offsets[i] < 0) return G4_ERR_INVALID_ARG;
    if (slots[i] < 0 || slots[i] >= c.max_batch || used[slots[i]]) return G4_ERR_INVALID_ARG;
    used[slots[i]] = 1;
    if (start_pos[i] < 0) return G4_ERR_INVALID_ARG;
    if ((int64_t)start_pos[i] + len[i] > c.max_context) return G4_ERR_CONTEXT_OVERFLOW;
    order[i] = i;
  }
  DEVICE_GUARD(h->device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (h->page_table) {  // pages for every prompt position, all or none
    long extra = 0;
    for (int i = 0; i < n_seq; ++i)
      extra += std::max(0, cdiv(start_pos[i] + len[i], 1 << h->page_shift) - h->slot_pages[slots[i]]);
    if (extra > (long)h->free_pages.size()) return G4_ERR_OOM;
    for (int i = 0; i < n_seq; ++i) TRY(kv_reserve_impl(h, st, slots[i], start_pos[i] + len[i]));
  }
  auto upload = [&](const std::vector<int>& host) -> g4_status {
    if (h->pf_cap < host.size()) {
      if (h->pf_buf) { CK(cudaStreamSynchronize(st)); cudaFree(h->pf_buf); h->pf_buf = nullptr; h->pf_cap = 0; }
      CK(cudaMalloc(&h->pf_buf, host.size() * sizeof(int)));
      h->pf_cap = host.size();
    }
    CK(cudaMemcpyAsync(h->pf_buf, host.data(), host.size() * sizeof(int), cudaMemcpyHostToDevice, st));
    CK(cudaStreamSynchronize(st));  // the host staging vector goes out of scope afterwards
    return G4_OK;
  };
  auto copy_out = [&](int q, int row, bool with_logits) -> g4_status {
    CK(cudaMemcpyAsync(d_next_ids + q, h->step_next + row, sizeof(int), cudaMemcpyDeviceToDevice, st));
    if (with_logits)
      CK(cudaMemcpyAsync(d_logits + (size_t)q * c.vocab, h->step_logits + (size_t)row * c.vocab,
                         (size_t)c.vocab * sizeof(float), cudaMemcpyDeviceToDevice, st));
    return G4_OK;
  };
  if (!h->trace) {
    // Blocks of up to kPrefillRows rows, sequence by sequence, positions ascending: each block
    // is one step whose K/V rows are all written before its attention, so a row sees the keys
    // of the earlier rows of its sequence in the same block.
    int total = 0;
    for (int i = 0; i < n_seq; ++i) total += len[i];
    const int n_blocks = (total + kPrefillRows - 1) / kPrefillRows;
    // [slots | positions | token indices] of all rows, then per block the rows that end a
    // sequence: [kept row index | slot | position] x kPrefillRows
    std::vector<int> host((size_t)3 * total + (size_t)n_blocks * 3 * kPrefillRows, 0);
    std::vector<int> last(n_seq);
    for (int i = 0, r = 0; i < n_seq; ++i) {
      for (int t = 0; t < len[i]; ++t, ++r) {
        host[(size_t)0 * total + r] = slots[i];
        host[(size_t)1 * total + r] = start_pos[i] + t;
        host[(size_t)2 * total + r] = offsets[i] + t;
      }
      last[i] = r - 1;  // the sequence's final row
    }
    std::vector<std::vector<int>> kept(n_blocks);  // sequences whose final row is in the block
    for (int i = 0; i < n_seq; ++i) kept[last[i] / kPrefillRows].push_back(i);
    for (int k = 0; k < n_blocks; ++k) {
      int* kb = host.data() + (size_t)3 * total + (size_t)k * 3 * kPrefillRows;
      for (size_t j = 0; j < kept[k].size(); ++j) {
        const int i = kept[k][j];
        kb[j] = last[i] - k * kPrefillRows;
        kb[kPrefillRows + j] = slots[i];
        kb[2 * kPrefillRows + j] = start_pos[i] + len[i] - 1;
      }
    }
    TRY(upload(host));
    for (int k = 0; k < n_blocks; ++k) {
      const int r0 = k * kPrefillRows, n = std::min(kPrefillRows, total - r0);
      const int* kb = h->pf_buf + (size_t)3 * total + (size_t)k * 3 * kPrefillRows;
      // compaction needs a K/V-free tail after layer 0; otherwise every row runs to the end
      const bool tail = h->l_tail > 0 && h->l_tail < c.num_layers;
      const int n_keep = (int)kept[k].size();
      float* lg = (d_logits && n_keep > 0) ? h->step_logits : nullptr;
      TRY(run_step(h, st, n, h->pf_buf + r0, d_tokens, h->pf_buf + (size_t)2 * total + r0, h->pf_buf + (size_t)total + r0,
                   h->step_next, lg, nullptr, true, kb, kb + kPrefillRows, kb + 2 * kPrefillRows, tail ? n_keep : -1));
      // rows kept past the K/V layers come out in kept order (ascending rows); without a
      // compaction (no K/V-free tail) they stay at their block rows
      const bool compacted = tail && n_keep < n;
      for (int j = 0; j < n_keep; ++j) {
        const int i = kept[k][j];
        TRY(copy_out(i, compacted ? j : last[i] - r0, d_logits != nullptr));
      }
    }
    return G4_OK;
  }
  // With a per-layer trace set: one decode step per prompt position (every active sequence
  // one row), so the trace rows stay the sequences' rows.
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return len[a] > len[b]; });
  const int T = len[order[0]];
  // per step t: slots, positions, token indices of the active prefix of `order`
  std::vector<int> host((size_t)3 * T * n_seq, 0);
  std::vector<int> n_act(T);
  for (int t = 0; t < T; ++t) {
    int n = 0;
    for (int i = 0; i < n_seq; ++i) {
      const int q = order[i];
      if (len[q] <= t) break;
      host[((size_t)0 * T + t) * n_seq + n] = slots[q];
      host[((size_t)1 * T + t) * n_seq + n] = start_pos[q] + t;
      host[((size_t)2 * T + t) * n_seq + n] = offsets[q] + t;
      ++n;
    }
    n_act[t] = n;
  }
  TRY(upload(host));
  for (int t = 0; t < T; ++t) {
    const int n = n_act[t];
    const int* ds = h->pf_buf + ((size_t)0 * T + t) * n_seq;
    const int* dp = h->pf_buf + ((size_t)1 * T + t) * n_seq;
    const int* di = h->pf_buf + ((size_t)2 * T + t) * n_seq;
    const int n_next = t + 1 < T ? n_act[t + 1] : 0;  // sequences finishing now: [n_next, n)
    float* lg = (d_logits && n_next < n) ? h->step_logits : nullptr;
    TRY(run_step(h, st, n, ds, d_tokens, di, dp, h->step_next, lg));
    for (int i = n_next; i < n; ++i) TRY(copy_out(order[i], i, d_logits != nullptr));
  }
  return G4_OK;
}

g4_status g4_profile_step(g4_handle* h, g4_stream stream, int32_t n_seq, const int32_t* d_slots,
                          const int32_t* d_tokens, const int32_t* d_positions, int32_t* d_next_ids, float* d_logits,
                          int32_t repeats, g4_phase_stat* stats, int32_t max_stats, int32_t* n_stats) {
  if (!h || !d_slots || !d_tokens || !d_positions || !d_next_ids || !stats || !n_stats || repeats < 1)
    return G4_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > h->cfg.max_batch) return G4_ERR_INVALID_ARG;
  DEVICE_GUARD(h->device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (h->mega_ok && h->mega_on && n_seq <= 2) {
    // persistent step: per-phase durations from the %globaltimer stamps CTA 0 takes after
    // every grid barrier (phase k ends when barrier k releases)
    std::map<std::string, g4_phase_stat> agg;
    std::vector<std::string> order;
    std::vector<unsigned long long> ts(h->mega_n + 1);
    for (int r = 0; r < repeats; ++r) {
      TRY(run_step_mega(h, st, n_seq, d_slots, d_tokens, nullptr, d_positions, d_next_ids, d_logits, true));
      CK(cudaMemcpyAsync(ts.data(), h->mega_stamps, ts.size() * 8, cudaMemcpyDeviceToHost, st));
      CK(cudaStreamSynchronize(st));
      for (int p = 0; p < h->mega_n; ++p) {
        const std::string& nm = h->mega_names[p];
        auto it = agg.find(nm);
        if (it == agg.end()) {
          g4_phase_stat z{};
          snprintf(z.name, sizeof z.name, "%s", nm.c_str());
          it = agg.emplace(nm, z).first;
          order.push_back(nm);
        }
        it->second.launches += 1;
        it->second.ms_total += (double)(ts[p + 1] - ts[p]) * 1e-6;
      }
    }
    int k = 0;
    for (const std::string& nm : order) {
      if (k >= max_stats) break;
      stats[k++] = agg[nm];
    }
    *n_stats = k;
    return G4_OK;
  }
  Prof prof;
  prof.st = st;
  float* saved_trace = h->trace;
  h->trace = nullptr;
  g4_status s = G4_OK;
  for (int r = 0; r < repeats && s == G4_OK; ++r)
    s = run_step(h, st, n_seq, d_slots, d_tokens, nullptr, d_positions, d_next_ids, d_logits, &prof);
  h->trace = saved_trace;
  if (s != G4_OK) return s;
  CK(cudaStreamSynchronize(st));
  std::vector<std::string> order;
  std::map<std::string, g4_phase_stat> agg;
  for (const Prof::Rec& r : prof.recs) {
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, r.a, r.b));
    auto it = agg.find(r.name);
    if (it == agg.end()) {
      g4_phase_stat z{};
      snprintf(z.name, sizeof z.name, "%s", r.name.c_str());
      it = agg.emplace(r.name, z).first;
      order.push_back(r.name);
    }
    it->second.launches += 1;
    it->second.ms_total += ms;
    it->second.bytes_total += r.bytes;
  }
  int k = 0;
  for (const std::string& nm : order) {
    if (k >= max_stats) break;
    stats[k++] = agg[nm];
  }
  *n_stats = k;
  return G4_OK;
}

g4_status g4_timeout_probe(g4_handle* h, g4_stream stream, int64_t wait_ns) {
  if (!h || wait_ns < 0 || wait_ns > 2000000000LL) return G4_ERR_INVALID_ARG;
  DEVICE_GUARD(h->device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!h->probe_flag) {
    TRY(dalloc(h, &h->probe_flag, 1));
    CK(cudaMemsetAsync(h->probe_flag, 0, sizeof(int), st));
  }
  probe_wait_kernel<<<1, 32, 0, st>>>(h->probe_flag, (unsigned long long)wait_ns, h->err);
  CK(cudaGetLastError());
  return G4_OK;
}

g4_status g4_get_device_error(g4_handle* h, g4_stream stream, int32_t* word_out) {
  if (!h) return G4_ERR_INVALID_ARG;
  DEVICE_GUARD(h->device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int w = 0;
  CK(cudaMemcpyAsync(&w, h->err, sizeof(int), cudaMemcpyDeviceToHost, st));
  CK(cudaMemsetAsync(h->err, 0, sizeof(int), st));
  CK(cudaStreamSynchronize(st));
  if (word_out) *word_out = w;
  if (w & G4_DEV_TIMEOUT) return G4_ERR_TIMEOUT;
  return w ? G4_ERR_DEVICE_CHECK : G4_OK;
}

// ------------------------------------------------------------------------ standalone ops
struct g4_linear_op {
  g4_handle h;  // owns the allocations
  Lin lin;
};

g4_status g4_linear_create(int device, int32_t weight_format, int32_t n_out, int32_t n_in, const void* d_w,
                           const void* d_scales, g4_linear_op** out) {
  if (!out || !d_w || n_out < 1 || n_in < 32 || n_in % 32) return G4_ERR_INVALID_ARG;
  if (weight_format != G4_BF16 && weight_format != G4_W4A16) return G4_ERR_INVALID_ARG;
  if (weight_format == G4_W4A16 && !d_scales) return G4_ERR_INVALID_ARG;
  *out = nullptr;
  DEVICE_GUARD(device);
  init_kernel_attrs(device);
  g4_linear_op* op = new g4_linear_op();
  op->h.device = device;
  cudaDeviceGetAttribute(&op->h.sms, cudaDevAttrMultiProcessorCount, device);
  cudaStream_t st = nullptr;
  CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
  std::vector<RbSrc> keep;
  g4_status s = build_lin(&op->h, weight_format, n_in, {{d_w, d_scales, n_out}}, false, &op->lin, st, keep);
  if (s == G4_OK) {
    plan_lin(op->lin, op->h.sms, false);
    size_t part = (size_t)op->lin.ksplit * kMaxNB * op->lin.n_rb * 32;
    size_t cnt = (size_t)op->lin.n_rb * op->lin.ksplit + 1;
    int ks, kbps;
    tc_plan(op->lin, op->h.sms, false, &ks, &kbps);
    cnt = std::max(cnt, (size_t)(op->lin.n_rb / 4) + 1);
    s = dalloc(&op->h, &op->h.gemv_part, part);
    if (s == G4_OK) s = dalloc(&op->h, &op->h.gemv_cnt, cnt);
    if (s == G4_OK && !cuda_ok(cudaMemsetAsync(op->h.gemv_cnt, 0, cnt * 4, st), "memset")) s = G4_ERR_CUDA;
    if (s == G4_OK) s = dalloc(&op->h, &op->h.xt, (size_t)tc_nkb(op->lin) * 2 * 64 * 128);
    if (s == G4_OK) s = dalloc(&op->h, &op->h.tc_part, (size_t)ks * 64 * (op->lin.n_rb / 4) * 128);
    if (s == G4_OK) s = dalloc(&op->h, &op->h.err, 1);
    if (s == G4_OK) s = dalloc(&op->h, &op->h.sg_ctr, (size_t)2 * kSgMaxParts);
    if (s == G4_OK && !cuda_ok(cudaMemsetAsync(op->h.sg_ctr, 0, 2 * kSgMaxParts * sizeof(unsigned), st), "memset"))
      s = G4_ERR_CUDA;
    if (s == G4_OK && !cuda_ok(cudaMemsetAsync(op->h.err, 0, 4, st), "memset")) s = G4_ERR_CUDA;
  }
  cudaStreamSynchronize(st);
  cudaStreamDestroy(st);
  if (s != G4_OK) {
    for (void* p : op->h.allocs) cudaFree(p);
    delete op;
    return s;
  }
  *out = op;
  return G4_OK;
}

g4_status g4_linear_forward(g4_linear_op* op, g4_stream stream, int32_t n_rows, const float* d_x, float* d_y) {
  if (!op || !d_x || !d_y || n_rows < 1 || n_rows > 64) return G4_ERR_INVALID_ARG;
  DEVICE_GUARD(op->h.device);
  GemvIO io;
  io.pro = PRO_PLAIN;
  io.x_in = d_x;
  io.x_stride = op->lin.K;
  io.y = d_y;
  io.y_stride = op->lin.n_valid;
  Scratch s{op->h.gemv_part, op->h.gemv_cnt, nullptr, nullptr, op->h.err};
  TcScratch tc{op->h.xt, op->h.tc_part, op->h.gemv_cnt, nullptr, nullptr, op->h.err};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (n_rows <= kMaxNB && gemv_staged_on()) {  // the decode step's projection kernel, one K slice
    StagedIn in;
    in.x = d_x;
    in.x_stride = op->lin.K;
    StagedOut out{d_y, op->lin.n_valid, 0, nullptr};
    if (run_staged(op->lin, in, out, n_rows, 0.f, op->h.err, op->h.sg_ctr, op->h.sms, st, true)) {
      CK(cudaGetLastError());
      return G4_OK;
    }
  }
  run_gemv(op->lin, EPI_STORE, io, n_rows, 0.f, s, op->h.sms, st, &tc);
  CK(cudaGetLastError());
  return G4_OK;
}

void g4_linear_free(g4_linear_op* op) {
  if (!op) return;
  DeviceGuard dg(op->h.device);
  cudaDeviceSynchronize();
  for (void* p : op->h.allocs) cudaFree(p);
  delete op;
}

// Per-device scratch of the standalone argmax, grown on demand and kept until exit.
namespace {
struct ArgmaxScratch {
  float* pv = nullptr;
  int* pi = nullptr;
  unsigned* cnt = nullptr;
  size_t cap = 0;
};
std::mutex g_am_mu;
std::map<int, ArgmaxScratch> g_am;
}  // namespace

g4_status g4_argmax_rows(int device, g4_stream stream, int32_t n_rows, int32_t n_cols, const float* d_logits,
                         int32_t* d_ids) {
  if (!d_logits || !d_ids || n_rows < 1 || n_rows > 64 || n_cols < 1) return G4_ERR_INVALID_ARG;
  DEVICE_GUARD(device);
  const int chunk = 4096;
  const int nchunk = cdiv(n_cols, chunk);
  const size_t need = (size_t)n_rows * nchunk;
  ArgmaxScratch* sc;
  {
    std::lock_guard<std::mutex> lk(g_am_mu);
    sc = &g_am[device];
    if (sc->cap < need) {
      CK(cudaDeviceSynchronize());
      cudaFree(sc->pv);
      cudaFree(sc->pi);
      cudaFree(sc->cnt);
      *sc = ArgmaxScratch{};
      CK(cudaMalloc(&sc->pv, need * sizeof(float)));
      CK(cudaMalloc(&sc->pi, need * sizeof(int)));
      CK(cudaMalloc(&sc->cnt, 64 * sizeof(unsigned)));
      CK(cudaMemset(sc->cnt, 0, 64 * sizeof(unsigned)));
      sc->cap = need;
    }
  }
  argmax_rows_kernel<<<dim3(nchunk, n_rows), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      d_logits, n_cols, chunk, sc->pv, sc->pi, sc->cnt, d_ids);
  CK(cudaGetLastError());
  return G4_OK;
}

// ---------------------------------------------------------------- argmax without allocation
// Scratch of the allocation-free argmax: per-block partial values and indices for up to
// kStaticArgmaxRows rows x kStaticArgmaxChunks column chunks, and one counter per row.
// Every GPU that loads the library holds this array until the process exits.
constexpr int kStaticArgmaxRows = 64;
constexpr int kStaticArgmaxChunks = 256;
constexpr int kStaticArgmaxChunk = 4096;
struct StaticArgmaxScratch {
  float pv[kStaticArgmaxRows * kStaticArgmaxChunks];
  int pi[kStaticArgmaxRows * kStaticArgmaxChunks];
  unsigned cnt[kStaticArgmaxRows];
};
static __device__ __align__(256) StaticArgmaxScratch g4_static_argmax_scratch;

namespace {
std::mutex g_static_mu;
std::map<int, StaticArgmaxScratch*> g_static_ptr;  // device -> device address of the array
}  // namespace

g4_status g4_argmax_rows_static(int device, g4_stream stream, int32_t n_rows, int32_t n_cols,
                                const float* d_logits, int32_t* d_ids) {
  if (!d_logits || !d_ids || n_rows < 1 || n_cols < 1) return G4_ERR_INVALID_ARG;
  const int nchunk = cdiv(n_cols, kStaticArgmaxChunk);
  if (n_rows > kStaticArgmaxRows || nchunk > kStaticArgmaxChunks) {
    g_last_cuda = "g4_argmax_rows_static: at most 64 rows and 1,048,576 columns";
    return G4_ERR_INVALID_ARG;
  }
  DEVICE_GUARD(device);
  StaticArgmaxScratch* sc = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_static_mu);
    auto it = g_static_ptr.find(device);
    if (it == g_static_ptr.end()) {
      // The array's host-side name is not a device address: look the address up once per
      // device, with that device current.
      void* p = nullptr;
      CK(cudaGetSymbolAddress(&p, g4_static_argmax_scratch));
      it = g_static_ptr.emplace(device, static_cast<StaticArgmaxScratch*>(p)).first;
    }
    sc = it->second;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // counters must start at zero (an earlier call may have been cut short)
  CK(cudaMemsetAsync(sc->cnt, 0, sizeof(unsigned) * n_rows, st));
  argmax_rows_kernel<<<dim3(nchunk, n_rows), 256, 0, st>>>(d_logits, n_cols, kStaticArgmaxChunk, sc->pv, sc->pi,
                                                           sc->cnt, d_ids);
  CK(cudaGetLastError());
  return G4_OK;
}

}  // extern "C"
