// Persistent decode step for 1-2 sequences: one cooperative launch (one CTA per SM) runs the
// whole step as a static program of phases separated by grid barriers, in place of the ~250
// kernel boundaries of the launch-per-phase path.
//
// Phases (the same arithmetic as the launch-per-phase path, see g4.cu):
//   PMP      pr parts = W_pmp (E[t] sqrt H)                       (K slices -> partials)
//   PLE      ple_l = (RMSNorm(sum parts(pr_l) H^-1/2) g + T_ple[t]_l sqrt P) / sqrt 2
//   GEMV     y = W f(x) with f one of: plain; RMSNorm; residual update x = (x + RMSNorm(sum
//            of the branch's K-slice partials) g) lambda, then RMSNorm; embedding gather
//            (x0 = E[t] sqrt H), then RMSNorm.  Output: final rows (with the GeGLU / PLE
//            epilogue) or raw K-slice partials, which the next residual update sums in
//            slice order.
//   ATTN     flash-decode units (attn_unit), two per CTA (one per 128-thread half; one for
//            head dim 512)
//   LMHEAD   final residual + RMSNorm, logits rows, running argmax per CTA (a projection
//            phase with an argmax epilogue)
//   ARGMAX   CTA 0 reduces the per-CTA argmax partials
// Units of a projection phase are (row group, K slice of spu supergroups), dealt round-robin
// to the CTAs; the CTA's eight warps share each unit's tiles.  Their weights arrive through
// the shared-memory weight ring (see MegaRing below).  The grid barrier is a monotonically
// increasing counter (cleared before the launch); its wait is bounded: on expiry a CTA sets
// the timeout bit and the abort flag, and every CTA leaves at its next wait.
// Visibility: data written by other CTAs earlier in the launch is read only through L2
// (cp.async.cg, ld.global.cg) or after the barrier's acquire fence, never from a possibly
// stale L1 line.
#pragma once
#include "attn.cuh"
#include "common.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"

namespace g4 {

constexpr int kMegaThreads = 256;
constexpr int kMegaWarps = kMegaThreads / 32;
static_assert(kMegaWarps == 8, "projection items give warp w tile w of each supergroup");
constexpr unsigned long long kBarrierTimeoutNs = 2000000000ull;  // 2 s
constexpr int kPhaseBufs = 4;  // phase descriptors p .. p + 3 staged in shared memory

enum { PH_PMP = 0, PH_PLE = 1, PH_GEMV = 2, PH_ATTN = 3, PH_LMHEAD = 4, PH_ARGMAX = 5 };
enum { IN_PLAIN = 0, IN_NORM = 2, IN_RESID = 3, IN_EMBED = 4, IN_EMBED_NORM = 5 };

struct __align__(16) MegaPhase {
  int type;
  // ---- projection
  const uint4* qw;
  const uint4* sc;
  int fmt, R, n_rb, tiles, S, K, n_valid;
  int spu, ksplit, n_units, chunk_sg;  // units: (row group, K slice of spu supergroups)
  // input
  int in_mode;
  const float* x_in;       // IN_PLAIN slice source / IN_NORM / IN_RESID residual
  int x_stride;            // row stride of x_in
  const float* r_in;       // IN_RESID: branch partial slices (summed in slice order)
  int r_parts;
  long r_part_stride;
  int r_stride;
  const __nv_bfloat16* g_r;
  float lambda;
  const __nv_bfloat16* g_a;
  float* x_out;            // IN_RESID / IN_EMBED*: the new residual (CTA 0 writes it)
  int trace_x;             // >= 0: the new residual is the stream after layer trace_x
  int trace_attn;          // >= 0: copy the attention output of layer trace_attn (IN_PLAIN phase)
  int trace_attn_width;
  // output
  float* y;
  int y_stride;
  long y_part_stride;      // ksplit > 1: partial slice s at y + s * y_part_stride
  int epi;                 // EPI_STORE / EPI_GEGLU / EPI_PLE (ksplit == 1)
  const float* ple;        // EPI_PLE
  int ple_stride;
  // ---- attention
  AttnArgs attn;
  int attn_d, attn_hpc, attn_units;
  // ---- PLE build
  int L, P;
  const float* pr_parts;
  int pr_nparts;
  long pr_part_stride;
  const __nv_bfloat16* g_ppn;
  const __nv_bfloat16* ple_table;
  float* ple_out;
  float inv_sqrt_h, inv_sqrt2, sqrt_p;
};

struct MegaArgs {
  const MegaPhase* phases;
  int n_phases;
  int nb;
  const int* slots;
  const int* positions;
  const int* tokens;
  const int* tok_idx;
  const __nv_bfloat16* embed;
  int H, V;
  float sqrt_h, eps;
  unsigned* barrier;     // [0] counter, [1] abort flag
  float* am_val;         // [nb][gridDim.x]
  int* am_idx;
  int* next_ids;
  float* logits;
  int logits_stride;
  int* err;
  unsigned long long* stamps;  // optional [n_phases + 1] %globaltimer after each phase (CTA 0)
  float* trace;                // optional per-layer trace (layout of g4_set_trace)
  int trace_stride, max_batch;
};

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier number `k` (0-based).  Returns false when the step was aborted.  One thread
// per CTA polls the counter without sleeping (each poll is an L2 round trip); every 256 polls
// it checks the abort flag and the %globaltimer deadline.
__device__ __forceinline__ bool grid_sync(const MegaArgs& a, unsigned k, int* abort_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned* ctr = a.barrier;
    volatile unsigned* abort_g = a.barrier + 1;
    __threadfence();
    red_release_add(ctr, 1u);
    const unsigned target = (k + 1) * gridDim.x;
    uint32_t it = 0;
    unsigned long long t0 = 0;
    int ab = 0;
    while (ld_acquire(ctr) < target) {
      if ((++it & 255u) == 0) {
        if (*abort_g) { ab = 1; break; }
        const unsigned long long now = globaltimer_ns();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > kBarrierTimeoutNs) {
          set_err(a.err, G4_DEV_TIMEOUT);
          *abort_g = 1u;
          ab = 1;
          break;
        }
      }
    }
    __threadfence();  // acquire side: later reads of this CTA see every CTA's phase writes
    *abort_s = ab;
  }
  cp_async_wait_all();  // descriptor copies issued before the barrier
  __syncthreads();
  return *abort_s == 0;
}

template <int NB>
__device__ __forceinline__ int mega_token(const MegaArgs& a, int b) {
  int t = a.tok_idx ? a.tokens[a.tok_idx[b]] : a.tokens[b];
  if (t < 0 || t >= a.V) t = 0;  // the error bit is raised once, by phase 0
  return t;
}

// Shared-memory carve of a whole-vector phase (floats): xf [NB][K] | rf [NB][K] | residual
// branch partials [r_parts][NB][K] | gains g_r, g_a (2 K bf16) | red [32 NB] | wred.
__host__ __device__ constexpr size_t full_rf(int nb, int K) { return (size_t)nb * K; }
__host__ __device__ constexpr size_t full_rp(int nb, int K) { return (size_t)2 * nb * K; }
__host__ __device__ constexpr size_t full_gain(int nb, int K, int r_parts) { return (size_t)(2 + r_parts) * nb * K; }
__host__ __device__ constexpr size_t full_red(int nb, int K, int r_parts) { return full_gain(nb, K, r_parts) + K; }

// Whole-vector prologue (IN_NORM / IN_RESID / IN_EMBED*): xf[b][0..K) in smem.  Rows, the
// residual branch's K-slice partials and both gain vectors are staged with one wave of
// cp.async, then reduced in shared memory (partials summed in slice order).  Descriptor fields
// are read once into registers: the loops below store to shared memory, which the compiler
// cannot separate from the shared-memory descriptor.
template <int NB>
__device__ void mega_full_input(const MegaArgs& a, const MegaPhase& ph, float* smem) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int K = ph.K, c4 = K / 4, nb = a.nb, in_mode = ph.in_mode, r_parts = ph.r_parts;
  const bool embed = in_mode == IN_EMBED || in_mode == IN_EMBED_NORM;
  const bool resid = in_mode == IN_RESID;
  const float* x_in = ph.x_in;
  const int x_stride = ph.x_stride;
  const float* r_in = ph.r_in;
  const long r_part_stride = ph.r_part_stride;
  const int r_stride = ph.r_stride;
  const __nv_bfloat16* g_r = ph.g_r;
  const __nv_bfloat16* g_a = in_mode != IN_EMBED ? ph.g_a : nullptr;
  const float lambda = ph.lambda;
  float* x_out = ph.x_out;
  const int trace_x = ph.trace_x;
  float* xf = smem;
  float* rf = smem + full_rf(NB, K);
  float* rparts = smem + full_rp(NB, K);
  __nv_bfloat16* gr_s = reinterpret_cast<__nv_bfloat16*>(smem + full_gain(NB, K, resid ? r_parts : 0));
  __nv_bfloat16* ga_s = gr_s + K;
  float* red = smem + full_red(NB, K, resid ? r_parts : 0);
  for (int i = tid; i < K / 8; i += nt) {
    if (resid) cp_async16(gr_s + 8 * i, g_r + 8 * i, true);
    if (g_a) cp_async16(ga_s + 8 * i, g_a + 8 * i, true);
  }
  if (embed) {
    const __nv_bfloat16* emb = a.embed;
    const float sh = a.sqrt_h;
    for (int i = tid; i < NB * (K / 8); i += nt) {
      const int b = i / (K / 8), c = i - b * (K / 8);
      float* dst = xf + b * K + 8 * c;
      if (b < nb) {
        const uint4 u = *reinterpret_cast<const uint4*>(emb + (size_t)mega_token<NB>(a, b) * K + 8 * c);
        dst[0] = bf16_lo(u.x) * sh; dst[1] = bf16_hi(u.x) * sh; dst[2] = bf16_lo(u.y) * sh; dst[3] = bf16_hi(u.y) * sh;
        dst[4] = bf16_lo(u.z) * sh; dst[5] = bf16_hi(u.z) * sh; dst[6] = bf16_lo(u.w) * sh; dst[7] = bf16_hi(u.w) * sh;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = 0.f;
      }
    }
  } else {
    for (int i = tid; i < NB * c4; i += nt) {
      const int b = i / c4, c = i - b * c4;
      const bool ok = b < nb;
      cp_async16(xf + b * K + 4 * c, ok ? x_in + (size_t)b * x_stride + 4 * c : x_in, ok);
      if (resid)
        for (int q = 0; q < r_parts; ++q)
          cp_async16(rparts + ((size_t)q * NB + b) * K + 4 * c,
                     ok ? r_in + q * r_part_stride + (size_t)b * r_stride + 4 * c : r_in, ok);
    }
  }
  cp_async_wait_all();
  __syncthreads();
  // Elementwise passes run on float4 groups (i = b * K/4 + c, three per thread at K = 1536,
  // NB = 2); per-row sums go to ss[0] / ss[1] by a select so they stay in registers.
  float4* xf4 = reinterpret_cast<float4*>(xf);
  if (resid) {
    float4* rf4 = reinterpret_cast<float4*>(rf);
    const float4* rp4 = reinterpret_cast<const float4*>(rparts);
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) ss[b] = 0.f;
    for (int i = tid; i < NB * c4; i += nt) {
      const int b = i / c4;
      float4 r = rp4[i];
      for (int q = 1; q < r_parts; ++q) {
        const float4 t = rp4[(size_t)q * NB * c4 + i];
        r.x += t.x; r.y += t.y; r.z += t.z; r.w += t.w;
      }
      rf4[i] = r;
      const float sq = r.x * r.x + r.y * r.y + r.z * r.z + r.w * r.w;
      if (NB == 1 || b == 0) ss[0] += sq; else ss[NB - 1] += sq;
    }
    block_sum<NB>(ss, red);
    float rd[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) rd[b] = rms_denom(ss[b], K, a.eps);
    for (int i = tid; i < NB * c4; i += nt) {
      const int b = i / c4, c = i - b * c4;
      const float d = (NB == 1 || b == 0) ? rd[0] : rd[NB - 1];
      const uint2 g = *reinterpret_cast<const uint2*>(gr_s + 4 * c);
      const float4 r = rf4[i];
      float4 x = xf4[i];
      x.x = (x.x + (r.x / d) * bf16_lo(g.x)) * lambda;
      x.y = (x.y + (r.y / d) * bf16_hi(g.x)) * lambda;
      x.z = (x.z + (r.z / d) * bf16_lo(g.y)) * lambda;
      x.w = (x.w + (r.w / d) * bf16_hi(g.y)) * lambda;
      xf4[i] = x;
    }
    __syncthreads();
  }
  if (blockIdx.x == 0 && x_out != nullptr && (resid || embed)) {
    float* tr = (a.trace && trace_x >= 0) ? a.trace + (size_t)(trace_x * 2 + 1) * a.max_batch * a.trace_stride : nullptr;
    for (int i = tid; i < nb * c4; i += nt) {
      const int b = i / c4, c = i - b * c4;
      const float4 v = xf4[i];
      *reinterpret_cast<float4*>(x_out + (size_t)b * x_stride + 4 * c) = v;
      if (tr) *reinterpret_cast<float4*>(tr + (size_t)b * a.trace_stride + 4 * c) = v;
    }
  }
  if (g_a != nullptr) {
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) ss[b] = 0.f;
    for (int i = tid; i < NB * c4; i += nt) {
      const int b = i / c4;
      const float4 x = xf4[i];
      const float sq = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
      if (NB == 1 || b == 0) ss[0] += sq; else ss[NB - 1] += sq;
    }
    block_sum<NB>(ss, red);
    float ad[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) ad[b] = rms_denom(ss[b], K, a.eps);
    for (int i = tid; i < NB * c4; i += nt) {
      const int b = i / c4, c = i - b * c4;
      const float d = (NB == 1 || b == 0) ? ad[0] : ad[NB - 1];
      const uint2 g = *reinterpret_cast<const uint2*>(ga_s + 4 * c);
      float4 x = xf4[i];
      x.x = (x.x / d) * bf16_lo(g.x);
      x.y = (x.y / d) * bf16_hi(g.x);
      x.z = (x.z / d) * bf16_lo(g.y);
      x.w = (x.w / d) * bf16_hi(g.y);
      xf4[i] = x;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------------------------
// Weight ring.  Weights never depend on activations, so each CTA streams the weights of its
// upcoming units into a shared-memory ring with 1-D bulk copies (cp.async.bulk, completion on
// an mbarrier) while earlier phases, barriers and prologues run; a projection phase then reads
// its weights from shared memory.  One thread (thread 0) is the producer; it runs at phase
// starts and after every consumed item, up to two phases ahead (the descriptors it can see).
// An item is one unit (row group x K slice) or, for units above kItemMax bytes, a chunk of
// chunk_sg supergroups of it; inside an item the layout is, per row block r, the tiles of its
// supergroups, then per row block r their scale vectors (W4A16).  Items are consumed in the
// order they are issued (the CTA's units of each phase in turn, all eight warps per item), and
// released one at a time, so every item that fits the ring can always be issued: no deadlock.
constexpr int kRingSlots = 8;
constexpr uint32_t kRingBytes = 128u * 1024u;
constexpr uint32_t kItemMax = 64u * 1024u;
constexpr uint32_t kTileBytes = 32 * 16;

struct MegaRing {
  uint64_t full[kRingSlots];     // item seq completes phase seq / kRingSlots of full[seq % kRingSlots]
  uint32_t off[kRingSlots];      // ring byte offset of item seq % kRingSlots
  uint32_t endpos[kRingSlots];   // monotonic end position of that item
  uint32_t head, tail;           // monotonic byte positions (issued end, released end)
  uint32_t issued, consumed;     // item counts
  int cur_p, cur_j, cur_c;       // producer cursor: phase, j-th unit of this CTA, chunk
  int dead;                      // a wait ran out: issue nothing more
};

__device__ __forceinline__ bool is_proj(int type) { return type == PH_GEMV || type == PH_PMP || type == PH_LMHEAD; }

// Geometry of the j-th unit of this CTA in phase ph (u = blockIdx.x + j * gridDim.x).
struct UnitGeo {
  int u, rg, ks, sg0, nsg, n_chunks;
};
__device__ __forceinline__ UnitGeo unit_geo(const MegaPhase& ph, int j) {
  UnitGeo g;
  g.u = blockIdx.x + j * gridDim.x;
  g.rg = g.u / ph.ksplit;
  g.ks = g.u - g.rg * ph.ksplit;
  g.sg0 = g.ks * ph.spu;
  g.nsg = min(ph.S, g.sg0 + ph.spu) - g.sg0;
  g.n_chunks = (g.nsg + ph.chunk_sg - 1) / ph.chunk_sg;
  return g;
}
__device__ __forceinline__ uint32_t sg_bytes(const MegaPhase& ph) {
  return 8 * kTileBytes + (ph.fmt == FMT_W4A16 ? kTileBytes : 0u);
}

// Producer (thread 0 only).  p_limit: last phase whose descriptor is in shared memory.
__device__ void ring_fill(const MegaArgs& a, MegaRing& R, unsigned char* ring, const MegaPhase* ph_s, int p_limit) {
  while (!R.dead && R.issued - R.consumed < (uint32_t)kRingSlots) {
    const int p = R.cur_p;
    if (p >= a.n_phases || p > p_limit) return;
    const MegaPhase& q = ph_s[p % kPhaseBufs];
    if (!is_proj(q.type)) { R.cur_p = p + 1; R.cur_j = 0; R.cur_c = 0; continue; }
    const UnitGeo g = unit_geo(q, R.cur_j);
    if (g.u >= q.n_units) { R.cur_p = p + 1; R.cur_j = 0; R.cur_c = 0; continue; }
    const int c0 = R.cur_c * q.chunk_sg;
    const int csz = min(q.chunk_sg, g.nsg - c0);
    const uint32_t qbytes = (uint32_t)csz * 8 * kTileBytes, sbytes = q.fmt == FMT_W4A16 ? (uint32_t)csz * kTileBytes : 0u;
    const uint32_t bytes = (uint32_t)q.R * (qbytes + sbytes);
    uint32_t start = R.head;
    if (start % kRingBytes + bytes > kRingBytes) start += kRingBytes - start % kRingBytes;  // wrap: skip the tail
    if (start + bytes - R.tail > kRingBytes) return;                                          // no room yet
    const int slot = R.issued % kRingSlots;
    const uint32_t off = start % kRingBytes;
    R.off[slot] = off;
    R.endpos[slot] = start + bytes;
    mbar_expect_tx(&R.full[slot], bytes);
    for (int r = 0; r < q.R; ++r) {
      const int rb = g.rg * q.R + r;
      const int s = g.sg0 + c0;
      bulk_g2s(ring + off + r * qbytes, q.qw + ((size_t)rb * q.tiles + (size_t)s * 8) * 32, qbytes, &R.full[slot]);
      if (sbytes) bulk_g2s(ring + off + q.R * qbytes + r * sbytes, q.sc + ((size_t)rb * q.S + s) * 32, sbytes, &R.full[slot]);
    }
    R.head = start + bytes;
    ++R.issued;
    if (++R.cur_c >= g.n_chunks) { R.cur_c = 0; ++R.cur_j; }
  }
}

// Bounded wait for item `seq` by each warp on its own (no CTA barrier).  On expiry the warp
// sets the timeout bit, the abort flag and R.dead; the caller reads R.dead after its next
// __syncthreads, so every thread of the CTA leaves together.
__device__ void ring_wait(const MegaArgs& a, MegaRing& R, uint32_t seq) {
  const int slot = seq % kRingSlots;
  const uint32_t parity = (seq / kRingSlots) & 1u;
  if (mbar_try(&R.full[slot], parity)) return;
  const unsigned long long t0 = globaltimer_ns();
  volatile unsigned* abort_g = a.barrier + 1;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(&R.full[slot], parity)) return;
    if ((it & 1023u) == 0 && (*abort_g || globaltimer_ns() - t0 > kBarrierTimeoutNs)) break;
  }
  if ((threadIdx.x & 31) == 0) {
    set_err(a.err, G4_DEV_TIMEOUT);
    *abort_g = 1u;
    R.dead = 1;
  }
}

// Leaving the launch (normally or on abort): wait, bounded, for every issued, unconsumed item so
// no bulk copy still writes shared memory when the CTA exits.
__device__ void ring_drain(MegaRing& R) {
  if (threadIdx.x != 0) return;
  for (uint32_t seq = R.consumed; seq != R.issued; ++seq) {
    const int slot = seq % kRingSlots;
    const uint32_t parity = (seq / kRingSlots) & 1u;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 0; !mbar_try(&R.full[slot], parity); ++it)
      if ((it & 1023u) == 0 && globaltimer_ns() - t0 > kBarrierTimeoutNs) break;
  }
  R.consumed = R.issued;
}

// Projection phase (GEMV, PMP, LMHEAD): the CTA's units in turn, all warps on each item; warp w
// takes the (supergroup, row block) pairs i = w, w + 8, ... of the item (i = s_local * R + r).
// Per unit, warp partial sums are reduced in fixed warp order; the epilogue writes final rows
// (plain / GeGLU / PLE), K-slice partials, or logits with a running per-CTA argmax.
template <int FMT, int NB>
__device__ __noinline__ bool mega_proj(const MegaArgs& a, const MegaPhase& ph, float* smem, MegaRing& R,
                                       unsigned char* ring, const MegaPhase* ph_s, int p) {
  constexpr int SGK = Fmt<FMT>::SGK, TK = Fmt<FMT>::TK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // descriptor fields in registers (the loops store to shared memory, where the descriptor lives)
  const int in_mode = ph.in_mode, K = ph.K, r_parts = ph.r_parts, nR = ph.R;
  const int spu = ph.spu, ksplit = ph.ksplit, n_units = ph.n_units, n_valid = ph.n_valid, epi = ph.epi;
  const float* x_in = ph.x_in;
  const int x_stride = ph.x_stride;
  float* y = ph.y;
  const int y_stride = ph.y_stride;
  const long y_part_stride = ph.y_part_stride;
  const float* ple = ph.ple;
  const int ple_stride = ph.ple_stride;
  const bool full_in = in_mode >= IN_NORM;
  const bool argmax = ph.type == PH_LMHEAD;
  const int slice = spu * SGK;
  // work region: full input [full_red + 32 NB] or slice [NB][slice], then wred [2][8][2 NB 32]
  float* xf = smem;
  float* xsl = smem;
  float* wred = smem + (full_in ? full_red(NB, K, in_mode == IN_RESID ? r_parts : 0) + 32 * NB : (size_t)NB * slice);
  const int my_units = (int)blockIdx.x < n_units ? (n_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  if (full_in && (my_units > 0 || (blockIdx.x == 0 && ph.x_out != nullptr))) mega_full_input<NB>(a, ph, smem);
  if (a.trace && ph.trace_attn >= 0 && blockIdx.x == 0) {
    const int tw = ph.trace_attn_width;
    float* tr = a.trace + (size_t)(ph.trace_attn * 2) * a.max_batch * a.trace_stride;
    for (int b = 0; b < a.nb; ++b)
      for (int k = threadIdx.x; k < tw; k += blockDim.x) tr[(size_t)b * a.trace_stride + k] = __ldcg(x_in + (size_t)b * x_stride + k);
  }
  float best_v[NB];
  int best_i[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) { best_v[b] = __int_as_float(0x7fc00000); best_i[b] = 0x7fffffff; }
  uint32_t seq = R.consumed;  // the same in every thread: advanced in lockstep below
  const uint32_t sgb = 8 * kTileBytes;
  for (int j = 0; j < my_units; ++j) {
    const UnitGeo g = unit_geo(ph, j);
    const float* xs;
    int xs_stride;
    if (full_in) {
      xs = xf + g.sg0 * SGK;
      xs_stride = K;
    } else {
      for (int i = threadIdx.x; i < NB * slice / 4; i += blockDim.x) {
        const int b = i / (slice / 4), c = i - b * (slice / 4), k = g.sg0 * SGK + 4 * c;
        const bool ok = b < a.nb && k < K;
        cp_async16(xsl + b * slice + 4 * c, ok ? x_in + (size_t)b * x_stride + k : x_in, ok);
      }
      cp_async_wait_all();
      __syncthreads();
      xs = xsl;
      xs_stride = slice;
    }
    float2 acc[2][NB];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = make_float2(0.f, 0.f);
    for (int c = 0; c < g.n_chunks; ++c) {
      ring_wait(a, R, seq);
      const bool live = !*reinterpret_cast<volatile int*>(&R.dead);
      const unsigned char* item = ring + R.off[seq % kRingSlots];
      const int c0 = c * ph.chunk_sg;
      const int csz = min(ph.chunk_sg, g.nsg - c0);
      const unsigned char* scb = item + (size_t)nR * csz * sgb;
      // warp w takes tile t = w of every (supergroup, row block) pair of the item: eight warps,
      // eight tiles per pair, so the item's tiles spread evenly over the CTA
      {
        const int t = warp;
        const float* xt = xs + c0 * SGK + t * TK;
        const int np = live ? csz * nR : 0;
        for (int i0 = 0; i0 < np; i0 += 4) {
          // four pairs' tiles and scales first, so their shared-memory loads overlap
          uint4 wv[4];
          uint32_t s2[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = min(i0 + u, np - 1);
            const int sl = i / nR, r = i - sl * nR;
            wv[u] = reinterpret_cast<const uint4*>(item + (size_t)(r * csz + sl) * sgb + t * kTileBytes)[lane];
            s2[u] = 0;
            if constexpr (FMT == FMT_W4A16) {
              const uint32_t sw = reinterpret_cast<const uint32_t*>(scb + (size_t)(r * csz + sl) * kTileBytes + lane * 16)[t >> 1];
              const uint32_t hh = (t & 1) ? (sw >> 16) : (sw & 0xFFFFu);
              s2[u] = hh | (hh << 16);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = i0 + u;
            if (i < np) {
              const int sl = i / nR, r = i - sl * nR;
              if (r == 0) tile_fma<FMT, NB>(wv[u], s2[u], xt + sl * SGK, xs_stride, acc[0]);
              else tile_fma<FMT, NB>(wv[u], s2[u], xt + sl * SGK, xs_stride, acc[1]);
            }
          }
        }
      }
      float* wr = wred + (size_t)(j & 1) * kMegaWarps * 2 * NB * 32;
      if (c + 1 == g.n_chunks) {
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int b = 0; b < NB; ++b) wr[warp * (2 * NB * 32) + (r * NB + b) * 32 + lane] = acc[r][b].x + acc[r][b].y;
      }
      __syncthreads();  // item consumed (and, on the last chunk, warp partials written)
      if (R.dead) return false;  // a wait ran out (read after the barrier: uniform)
      ++seq;
      if (threadIdx.x == 0) {
        R.consumed = seq;
        R.tail = R.endpos[(seq - 1) % kRingSlots];
        ring_fill(a, R, ring, ph_s, p + 2);
      }
    }
    if (warp == 0) {
      const float* wr = wred + (size_t)(j & 1) * kMegaWarps * 2 * NB * 32;
      float v[2][NB];
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float sacc = 0.f;
#pragma unroll
          for (int w = 0; w < kMegaWarps; ++w) sacc += wr[w * (2 * NB * 32) + (r * NB + b) * 32 + lane];
          v[r][b] = sacc;
        }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= a.nb) break;
        if (argmax) {
          const int n = g.rg * 32 + lane;
          if (n < n_valid) {
            if (a.logits) a.logits[(size_t)b * a.logits_stride + n] = v[0][b];
            if (argmax_better(v[0][b], n, best_v[b], best_i[b])) { best_v[b] = v[0][b]; best_i[b] = n; }
          }
        } else if (ksplit > 1) {
#pragma unroll
          for (int r = 0; r < 2; ++r)
            if (r < nR) y[g.ks * y_part_stride + (size_t)b * y_stride + (g.rg * nR + r) * 32 + lane] = v[r][b];
        } else if (epi == EPI_GEGLU) {
          const int n = g.rg * 32 + lane;  // row block 0 = gate rows, 1 = up rows
          if (n < n_valid) y[(size_t)b * y_stride + n] = gelu_tanh(v[0][b]) * v[1][b];
        } else {
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int row = (g.rg * nR + r) * 32 + lane;
            if (r >= nR || row >= n_valid) continue;
            float o = v[r][b];
            if (epi == EPI_PLE) o = gelu_tanh(o) * __ldcg(ple + (size_t)b * ple_stride + row);
            y[(size_t)b * y_stride + row] = o;
          }
        }
      }
    }
  }
  if (argmax && warp == 0) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      if (b >= a.nb) break;
      float v = best_v[b];
      int i = best_i[b];
      warp_argmax(v, i);
      if (lane == 0) {
        a.am_val[b * gridDim.x + blockIdx.x] = v;
        a.am_idx[b * gridDim.x + blockIdx.x] = i;
      }
    }
  }
  return true;
}

template <int NB>
__device__ void mega_ple(const MegaArgs& a, const MegaPhase& ph, float* smem) {
  const auto ph_P = ph.P;
  const auto ph_L = ph.L;
  const auto ph_pr_nparts = ph.pr_nparts;
  const auto ph_pr_parts = ph.pr_parts;
  const auto ph_pr_part_stride = ph.pr_part_stride;
  const auto ph_inv_sqrt_h = ph.inv_sqrt_h;
  const auto ph_ple_table = ph.ple_table;
  const auto ph_sqrt_p = ph.sqrt_p;
  const auto ph_ple_out = ph.ple_out;
  const auto ph_g_ppn = ph.g_ppn;
  const auto ph_inv_sqrt2 = ph.inv_sqrt2;
  // one (b, l) chunk of P per CTA iteration
  const int tid = threadIdx.x, nt = blockDim.x;
  float* v = smem;           // [P]
  float* red = smem + ph_P;  // [32]
  for (int c = blockIdx.x; c < a.nb * ph_L; c += gridDim.x) {
    const int b = c / ph_L, l = c - b * ph_L;
    const int t = mega_token<NB>(a, b);
    float ss[1] = {0.f};
    for (int i = tid; i < ph_P; i += nt) {
      float x = 0.f;
      for (int s = 0; s < ph_pr_nparts; ++s)
        x += __ldcg(ph_pr_parts + s * ph_pr_part_stride + (size_t)b * ph_L * ph_P + l * ph_P + i);
      x *= ph_inv_sqrt_h;
      v[i] = x;
      ss[0] += x * x;
    }
    block_sum<1>(ss, red);
    const float den = rms_denom(ss[0], ph_P, a.eps);
    for (int i = tid; i < ph_P; i += nt) {
      const float tok = bf16f(ph_ple_table[(size_t)t * ph_L * ph_P + l * ph_P + i]) * ph_sqrt_p;
      ph_ple_out[((size_t)b * ph_L + l) * ph_P + i] = ((v[i] / den) * bf16f(ph_g_ppn[i]) + tok) * ph_inv_sqrt2;
    }
    __syncthreads();
  }
}

// Attention units: two at a time on the CTA's two 128-thread halves (each with its own
// shared memory and named barrier), one at a time for head dim 512 (shared-memory budget).
template <int D>
__host__ __device__ constexpr int attn_halves() { return D >= 512 ? 1 : 2; }
template <int D>
__device__ __noinline__ void mega_attn_d(const MegaArgs& a, const MegaPhase& ph, unsigned char* smem) {
  constexpr int H = attn_halves<D>();
  const int half = threadIdx.x >> 7;
  if (half >= H) return;
  const int n_hg = ph.attn.nq;  // one query head per unit
  const int units = ph.attn_units, nsplit = ph.attn.nsplit;
  unsigned char* my = smem + half * attn_smem_bytes<D, 1>(ph.attn.nstage);
  for (int u0 = blockIdx.x * H; u0 < units; u0 += gridDim.x * H) {
    const int u = u0 + half;
    const int b = u / (nsplit * n_hg);
    if (u < units && b < a.nb) {
      AttnArgs aa = ph.attn;
      aa.slots = a.slots;
      aa.positions = a.positions;
      const int split = u % nsplit;
      const int hg = (u / nsplit) % n_hg;
      attn_unit<D, 1>(aa, split, hg, b, my, half * 128, 1 + half);
    }
  }
}

template <int NB>
__device__ void mega_argmax(const MegaArgs& a, float* smem) {
  if (blockIdx.x != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* rv = smem;
  int* ri = reinterpret_cast<int*>(smem + 32);
  for (int b = 0; b < a.nb; ++b) {
    float v = __int_as_float(0x7fc00000);
    int idx = 0x7fffffff;
    for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x) {
      const float cv = ldcg(a.am_val + b * gridDim.x + c);
      const int ci = __ldcg(a.am_idx + b * gridDim.x + c);
      if (argmax_better(cv, ci, v, idx)) { v = cv; idx = ci; }
    }
    warp_argmax(v, idx);
    if (lane == 0) { rv[warp] = v; ri[warp] = idx; }
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 1; w < kMegaWarps; ++w)
        if (argmax_better(rv[w], ri[w], rv[0], ri[0])) { rv[0] = rv[w]; ri[0] = ri[w]; }
      a.next_ids[b] = ri[0] == 0x7fffffff ? 0 : ri[0];
    }
    __syncthreads();
  }
}

// Stage phase descriptor p in shared memory with cp.async (no register round trip, so it can
// be issued just before a barrier without delaying the arrival; grid_sync waits for it).  The
// program is never written during the launch.  Reading descriptors from global memory inside
// a phase would cost an L2 round trip per field: the barrier's acquire invalidates L1.
__device__ __forceinline__ void load_phase(const MegaArgs& a, int p, MegaPhase* dst) {
  static_assert(sizeof(MegaPhase) % 16 == 0, "phase descriptor copied in 16-byte chunks");
  if (p >= a.n_phases) return;
  const char* src = reinterpret_cast<const char*>(a.phases + p);
  char* d = reinterpret_cast<char*>(dst);
  for (int i = threadIdx.x; i < (int)(sizeof(MegaPhase) / 16); i += blockDim.x) cp_async16(d + 16 * i, src + 16 * i, true);
}

template <int NB>
__global__ void __launch_bounds__(kMegaThreads, 1) mega_step_kernel(const MegaArgs a) {
  extern __shared__ __align__(128) unsigned char mdyn[];
  __shared__ int abort_s;
  __shared__ MegaPhase ph_s[kPhaseBufs];  // descriptors p .. p + 3
  __shared__ MegaRing ring_s;
  unsigned char* ring = mdyn;                                   // [kRingBytes] weight ring
  float* work = reinterpret_cast<float*>(mdyn + kRingBytes);    // per-phase work region
  if (blockIdx.x == 0 && threadIdx.x < a.nb) {
    const int t = a.tok_idx ? a.tokens[a.tok_idx[threadIdx.x]] : a.tokens[threadIdx.x];
    if (t < 0 || t >= a.V) set_err(a.err, G4_DEV_BAD_TOKEN);
  }
  if (a.stamps && blockIdx.x == 0 && threadIdx.x == 0) a.stamps[0] = globaltimer_ns();
  for (int q = 0; q < 3; ++q) load_phase(a, q, &ph_s[q]);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingSlots; ++i) mbar_init(&ring_s.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    ring_s.head = ring_s.tail = ring_s.issued = ring_s.consumed = 0;
    ring_s.cur_p = ring_s.cur_j = ring_s.cur_c = 0;
    ring_s.dead = 0;
  }
  cp_async_wait_all();
  __syncthreads();
  for (int p = 0; p < a.n_phases; ++p) {
    const MegaPhase& ph = ph_s[p % kPhaseBufs];
    if (threadIdx.x == 0) ring_fill(a, ring_s, ring, ph_s, p + 2);
    bool ok = true;
    switch (ph.type) {
      case PH_PMP:
      case PH_GEMV:
      case PH_LMHEAD:
        if (ph.fmt == FMT_W4A16) ok = mega_proj<FMT_W4A16, NB>(a, ph, work, ring_s, ring, ph_s, p);
        else ok = mega_proj<FMT_BF16, NB>(a, ph, work, ring_s, ring, ph_s, p);
        break;
      case PH_PLE:
        mega_ple<NB>(a, ph, work);
        break;
      case PH_ATTN:
        switch (ph.attn_d) {
          case 64: mega_attn_d<64>(a, ph, reinterpret_cast<unsigned char*>(work)); break;
          case 128: mega_attn_d<128>(a, ph, reinterpret_cast<unsigned char*>(work)); break;
          case 256: mega_attn_d<256>(a, ph, reinterpret_cast<unsigned char*>(work)); break;
          default: mega_attn_d<512>(a, ph, reinterpret_cast<unsigned char*>(work)); break;
        }
        break;
      case PH_ARGMAX:
        mega_argmax<NB>(a, work);
        break;
    }
    if (!ok) break;
    if (p + 1 < a.n_phases) {
      load_phase(a, p + 3, &ph_s[(p + 3) % kPhaseBufs]);  // buffer of phase p - 1: free
      if (!grid_sync(a, (unsigned)p, &abort_s)) break;
    }
    if (a.stamps && blockIdx.x == 0 && threadIdx.x == 0) a.stamps[p + 1] = globaltimer_ns();
  }
  __syncthreads();
  ring_drain(ring_s);
}

}  // namespace g4
