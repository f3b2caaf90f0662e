// Persistent decode step for 1-2 sequences: one cooperative launch runs the whole step as a
// static program of phases separated by grid barriers.  It removes the ~250 kernel
// boundaries of the launch-per-phase path, which at batch 1 cost more than the 1.87 GB of
// weights take to stream.
//
// Phases (the same arithmetic as the launch-per-phase path, see g4.cu):
//   PMP      pr parts = W_pmp (E[t] sqrt H)                       (K slices -> partials)
//   PLE      ple_l = (RMSNorm(sum parts(pr_l) H^-1/2) g + T_ple[t]_l sqrt P) / sqrt 2
//   GEMV     y = W f(x) with f one of: plain; RMSNorm; residual update x = (x + RMSNorm(sum
//            of the branch's K-slice partials) g) lambda, then RMSNorm; embedding gather
//            (x0 = E[t] sqrt H), then RMSNorm.  Output: final rows (with the GeGLU / PLE
//            epilogue) or raw K-slice partials, which the next residual update sums in
//            slice order.
//   ATTN     flash-decode units (attn_unit), two per CTA (one per 128-thread half)
//   LMHEAD   final residual + RMSNorm, logits rows, running argmax per CTA
//   ARGMAX   CTA 0 reduces the per-CTA argmax partials
// Units of a GEMV phase are (row group, K slice of spu supergroups); a CTA runs upc units
// at once with wpu warps each (upc * wpu = 8).  The grid barrier is a monotonically
// increasing counter (cleared before the launch); its wait is bounded: on expiry a CTA sets
// the timeout bit and the abort flag, and every CTA leaves at its next barrier.
// Visibility: data written by other CTAs earlier in the launch is read only through L2 (cp.async.cg,
// ld.global.cg) or after the barrier's acquire fence, never from a possibly stale L1 line.
#pragma once
#include "attn.cuh"
#include "common.cuh"
#include "gemv.cuh"

namespace g4 {

constexpr int kMegaThreads = 256;
constexpr int kMegaWarps = kMegaThreads / 32;
constexpr uint32_t kBarrierSpinLimit = 1u << 22;

enum { PH_PMP = 0, PH_PLE = 1, PH_GEMV = 2, PH_ATTN = 3, PH_LMHEAD = 4, PH_ARGMAX = 5 };
enum { IN_PLAIN = 0, IN_NORM = 2, IN_RESID = 3, IN_EMBED = 4, IN_EMBED_NORM = 5 };

struct MegaPhase {
  int type;
  // ---- projection
  const uint4* qw;
  const uint4* sc;
  int fmt, R, n_rb, tiles, S, K, n_valid;
  int spu, ksplit, wpu, upc, n_units;
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

// Grid barrier number `k` (0-based).  Returns false when the step was aborted.
__device__ __forceinline__ bool grid_sync(const MegaArgs& a, unsigned k, int* abort_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned* ctr = a.barrier;
    volatile unsigned* abort_g = a.barrier + 1;
    __threadfence();
    red_release_add(ctr, 1u);
    const unsigned target = (k + 1) * gridDim.x;
    uint32_t it = 0;
    int ab = 0;
    while (ld_acquire(ctr) < target) {
      if (*abort_g) { ab = 1; break; }
      if (++it > kBarrierSpinLimit) {
        set_err(a.err, G4_DEV_TIMEOUT);
        *abort_g = 1u;
        ab = 1;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();  // acquire side: later reads of this CTA see every CTA's phase writes
    *abort_s = ab;
  }
  __syncthreads();
  return *abort_s == 0;
}

template <int NB>
__device__ __forceinline__ int mega_token(const MegaArgs& a, int b) {
  int t = a.tok_idx ? a.tokens[a.tok_idx[b]] : a.tokens[b];
  if (t < 0 || t >= a.V) t = 0;  // the error bit is raised once, by phase 0
  return t;
}

// Whole-vector prologue (IN_NORM / IN_RESID / IN_EMBED*): xf[b][0..K) in smem.  Rows and the
// residual branch's K-slice partials are staged with one wave of cp.async, then reduced in
// shared memory (partials summed in slice order).
template <int NB>
__device__ void mega_full_input(const MegaArgs& a, const MegaPhase& ph, float* xf, float* rf, float* red) {
  const int tid = threadIdx.x, nt = blockDim.x, K = ph.K, c4 = K / 4;
  const bool embed = ph.in_mode == IN_EMBED || ph.in_mode == IN_EMBED_NORM;
  const bool resid = ph.in_mode == IN_RESID;
  float* rparts = rf + NB * K;  // [r_parts][NB][K]
  if (embed) {
    for (int i = tid; i < NB * (K / 8); i += nt) {
      const int b = i / (K / 8), c = i - b * (K / 8);
      float* dst = xf + b * K + 8 * c;
      if (b < a.nb) {
        const uint4 u = *reinterpret_cast<const uint4*>(a.embed + (size_t)mega_token<NB>(a, b) * K + 8 * c);
        const float sh = a.sqrt_h;
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
      const bool ok = b < a.nb;
      cp_async16(xf + b * K + 4 * c, ok ? ph.x_in + (size_t)b * ph.x_stride + 4 * c : ph.x_in, ok);
      if (resid)
        for (int q = 0; q < ph.r_parts; ++q)
          cp_async16(rparts + ((size_t)q * NB + b) * K + 4 * c,
                     ok ? ph.r_in + q * ph.r_part_stride + (size_t)b * ph.r_stride + 4 * c : ph.r_in, ok);
    }
    cp_async_wait_all();
  }
  __syncthreads();
  if (resid) {
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ss[b] = 0.f;
      for (int k = tid; k < K; k += nt) {
        float r = 0.f;
        for (int q = 0; q < ph.r_parts; ++q) r += rparts[((size_t)q * NB + b) * K + k];
        rf[b * K + k] = r;
        ss[b] += r * r;
      }
    }
    block_sum<NB>(ss, red);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float rd = rms_denom(ss[b], K, a.eps);
      for (int k = tid; k < K; k += nt)
        xf[b * K + k] = (xf[b * K + k] + (rf[b * K + k] / rd) * bf16f(ph.g_r[k])) * ph.lambda;
    }
    __syncthreads();
  }
  if (blockIdx.x == 0 && ph.x_out != nullptr && (resid || embed)) {
    for (int i = tid; i < a.nb * c4; i += nt) {
      const int b = i / c4, c = i - b * c4;
      *reinterpret_cast<float4*>(ph.x_out + (size_t)b * ph.x_stride + 4 * c) =
          *reinterpret_cast<const float4*>(xf + b * K + 4 * c);
      if (a.trace && ph.trace_x >= 0)
        *reinterpret_cast<float4*>(a.trace + ((size_t)(ph.trace_x * 2 + 1) * a.max_batch + b) * a.trace_stride + 4 * c) =
            *reinterpret_cast<const float4*>(xf + b * K + 4 * c);
    }
  }
  if (ph.in_mode != IN_EMBED && ph.g_a != nullptr) {
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ss[b] = 0.f;
      for (int k = tid; k < K; k += nt) ss[b] += xf[b * K + k] * xf[b * K + k];
    }
    block_sum<NB>(ss, red);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float ad = rms_denom(ss[b], K, a.eps);
      for (int k = tid; k < K; k += nt) xf[b * K + k] = (xf[b * K + k] / ad) * bf16f(ph.g_a[k]);
    }
  }
  __syncthreads();
}

template <int FMT, int NB>
__device__ void mega_gemv(const MegaArgs& a, const MegaPhase& ph, float* smem) {
  constexpr int SGK = Fmt<FMT>::SGK, TK = Fmt<FMT>::TK;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool full_in = ph.in_mode >= IN_NORM;
  const int slice = ph.spu * SGK;
  // full-input modes: xf [NB][K] | rf [NB][K] | r partial slices [r_parts][NB][K] | red | wred
  // slice mode:       xsl [upc][NB][slice] | wred
  float* xf = smem;
  float* rf = xf + NB * ph.K;
  float* red = rf + NB * ph.K + (ph.in_mode == IN_RESID ? ph.r_parts * NB * ph.K : 0);
  float* xsl = smem;
  float* wred = full_in ? red + 32 * NB : xsl + ph.upc * NB * slice;  // [8][2 * NB * 32]
  if (full_in) mega_full_input<NB>(a, ph, xf, rf, red);
  if (a.trace && ph.trace_attn >= 0 && blockIdx.x == 0) {
    for (int b = 0; b < a.nb; ++b)
      for (int k = threadIdx.x; k < ph.trace_attn_width; k += blockDim.x)
        a.trace[((size_t)(ph.trace_attn * 2) * a.max_batch + b) * a.trace_stride + k] =
            __ldcg(ph.x_in + (size_t)b * ph.x_stride + k);
  }
  const int slot = warp / ph.wpu, wi = warp % ph.wpu;
  const int n_batches = (ph.n_units + ph.upc - 1) / ph.upc;
  for (int bt = blockIdx.x; bt < n_batches; bt += gridDim.x) {
    const int u = bt * ph.upc + slot;
    const bool active = slot < ph.upc && u < ph.n_units;
    const int rg = active ? u / ph.ksplit : 0, ks = active ? u % ph.ksplit : 0;
    const int sg0 = ks * ph.spu, sg1 = min(ph.S, sg0 + ph.spu);
    const int k0 = sg0 * SGK;
    // issue this warp's first supergroup of weights before staging activations
    uint4 wbuf[2][8];
    uint4 sbuf[2];
    auto load_sg = [&](int s) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (r >= ph.R) break;
        const int rb = rg * ph.R + r;
        const uint4* base = ph.qw + ((size_t)rb * ph.tiles + (size_t)s * 8) * 32 + lane;
#pragma unroll
        for (int t = 0; t < 8; ++t) wbuf[r][t] = __ldg(base + t * 32);
        if constexpr (FMT == FMT_W4A16) sbuf[r] = __ldg(ph.sc + ((size_t)rb * ph.S + s) * 32 + lane);
      }
    };
    int sg = sg0 + wi;
    if (active && sg < sg1) load_sg(sg);
    // activation slice
    const float* xs;
    int xs_stride;
    if (full_in) {
      xs = xf + k0;
      xs_stride = ph.K;
    } else {
      float* my = xsl + (slot < ph.upc ? slot : 0) * NB * slice;
      const int tid_s = wi * 32 + lane, nt_s = ph.wpu * 32;
      if (slot < ph.upc) {
        for (int i = tid_s; i < NB * slice / 4; i += nt_s) {
          const int b = i / (slice / 4), c = i - b * (slice / 4), k = k0 + 4 * c;
          const bool ok = active && b < a.nb && k < ph.K;
          cp_async16(my + b * slice + 4 * c, ok ? ph.x_in + (size_t)b * ph.x_stride + k : ph.x_in, ok);
        }
      }
      cp_async_wait_all();
      xs = my;
      xs_stride = slice;
    }
    __syncthreads();
    float2 acc[2][NB];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = make_float2(0.f, 0.f);
    while (active && sg < sg1) {
      const float* xsg = xs + (sg - sg0) * SGK;
#pragma unroll
      for (int t = 0; t < 8; ++t) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          if (r >= ph.R) break;
          uint32_t s2 = 0;
          if constexpr (FMT == FMT_W4A16) {
            const uint32_t sw = (&sbuf[r].x)[t >> 1];
            const uint32_t hh = (t & 1) ? (sw >> 16) : (sw & 0xFFFFu);
            s2 = hh | (hh << 16);
          }
          tile_fma<FMT, NB>(wbuf[r][t], s2, xsg + t * TK, xs_stride, acc[r]);
        }
      }
      sg += ph.wpu;
      if (sg < sg1) load_sg(sg);
    }
    // reduce over the unit's warps
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) wred[warp * (2 * NB * 32) + (r * NB + b) * 32 + lane] = acc[r][b].x + acc[r][b].y;
    __syncthreads();
    if (active && wi == 0) {
      for (int r = 0; r < ph.R; ++r) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b >= a.nb) break;
          float v = 0.f;
          for (int w = 0; w < ph.wpu; ++w) v += wred[(slot * ph.wpu + w) * (2 * NB * 32) + (r * NB + b) * 32 + lane];
          const int row = (rg * ph.R + r) * 32 + lane;
          if (ph.ksplit > 1) {
            ph.y[ks * ph.y_part_stride + (size_t)b * ph.y_stride + row] = v;
          } else if (ph.epi == EPI_GEGLU) {
            if (r == 0) wred[(slot * ph.wpu) * (2 * NB * 32) + (0 * NB + b) * 32 + lane] = v;  // keep gate
            else {
              const float g = wred[(slot * ph.wpu) * (2 * NB * 32) + (0 * NB + b) * 32 + lane];
              const int n = rg * 32 + lane;
              if (n < ph.n_valid) ph.y[(size_t)b * ph.y_stride + n] = gelu_tanh(g) * v;
            }
          } else if (row < ph.n_valid) {
            if (ph.epi == EPI_PLE) v = gelu_tanh(v) * __ldcg(ph.ple + (size_t)b * ph.ple_stride + row);
            ph.y[(size_t)b * ph.y_stride + row] = v;
          }
        }
      }
    }
    __syncthreads();
  }
}

template <int NB>
__device__ void mega_ple(const MegaArgs& a, const MegaPhase& ph, float* smem) {
  // one (b, l) chunk of P per CTA iteration
  const int tid = threadIdx.x, nt = blockDim.x;
  float* v = smem;           // [P]
  float* red = smem + ph.P;  // [32]
  for (int c = blockIdx.x; c < a.nb * ph.L; c += gridDim.x) {
    const int b = c / ph.L, l = c - b * ph.L;
    const int t = mega_token<NB>(a, b);
    float ss[1] = {0.f};
    for (int i = tid; i < ph.P; i += nt) {
      float x = 0.f;
      for (int s = 0; s < ph.pr_nparts; ++s)
        x += __ldcg(ph.pr_parts + s * ph.pr_part_stride + (size_t)b * ph.L * ph.P + l * ph.P + i);
      x *= ph.inv_sqrt_h;
      v[i] = x;
      ss[0] += x * x;
    }
    block_sum<1>(ss, red);
    const float den = rms_denom(ss[0], ph.P, a.eps);
    for (int i = tid; i < ph.P; i += nt) {
      const float tok = bf16f(ph.ple_table[(size_t)t * ph.L * ph.P + l * ph.P + i]) * ph.sqrt_p;
      ph.ple_out[((size_t)b * ph.L + l) * ph.P + i] = ((v[i] / den) * bf16f(ph.g_ppn[i]) + tok) * ph.inv_sqrt2;
    }
    __syncthreads();
  }
}

template <int D>
__device__ void mega_attn_d(const MegaArgs& a, const MegaPhase& ph, unsigned char* smem) {
  // two units at a time: threads [0,128) and [128,256), each with its own smem and barrier
  const int half = threadIdx.x >> 7;
  const int n_hg = ph.attn.nq / ph.attn_hpc;
  unsigned char* my = smem + half * (ph.attn_hpc == 1 ? attn_smem_bytes<D, 1>(ph.attn.nstage)
                                                      : attn_smem_bytes<D, 8>(ph.attn.nstage));
  for (int u0 = blockIdx.x * 2; u0 < ph.attn_units; u0 += gridDim.x * 2) {
    const int u = u0 + half;
    const int b = u / (ph.attn.nsplit * n_hg);
    if (u < ph.attn_units && b < a.nb) {
      AttnArgs aa = ph.attn;
      aa.slots = a.slots;
      aa.positions = a.positions;
      const int split = u % ph.attn.nsplit;
      const int hg = (u / ph.attn.nsplit) % n_hg;
      if (ph.attn_hpc == 1) attn_unit<D, 1>(aa, split, hg, b, my, half * 128, 1 + half);
      else attn_unit<D, 8>(aa, split, hg, b, my, half * 128, 1 + half);
    }
  }
}

template <int NB>
__device__ void mega_lmhead(const MegaArgs& a, const MegaPhase& ph, float* smem) {
  // bf16 rows; every CTA holds the whole normalised input; running argmax per CTA
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* xf = smem;
  float* rf = xf + NB * ph.K;
  float* red = rf + NB * ph.K + ph.r_parts * NB * ph.K;
  float* wred = red + 32 * NB;  // [8][NB * 32]
  mega_full_input<NB>(a, ph, xf, rf, red);
  float best_v[NB];
  int best_i[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) { best_v[b] = __int_as_float(0x7fc00000); best_i[b] = 0x7fffffff; }
  const int n_rg = ph.n_rb;
  for (int rg = blockIdx.x; rg < n_rg; rg += gridDim.x) {
    float2 acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = make_float2(0.f, 0.f);
    constexpr int kMaxSgPerWarp = 4;  // K <= 2048 for the lm_head of this path
    uint4 w[kMaxSgPerWarp][8];
#pragma unroll
    for (int j = 0; j < kMaxSgPerWarp; ++j) {
      const int sg = warp + j * kMegaWarps;
      if (sg < ph.S) {
        const uint4* base = ph.qw + ((size_t)rg * ph.tiles + (size_t)sg * 8) * 32 + lane;
#pragma unroll
        for (int t = 0; t < 8; ++t) w[j][t] = __ldg(base + t * 32);
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxSgPerWarp; ++j) {
      const int sg = warp + j * kMegaWarps;
      if (sg < ph.S) {
#pragma unroll
        for (int t = 0; t < 8; ++t) tile_fma<FMT_BF16, NB>(w[j][t], 0u, xf + sg * 64 + t * 8, ph.K, acc);
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) wred[warp * NB * 32 + b * 32 + lane] = acc[b].x + acc[b].y;
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= a.nb) break;
        float v = 0.f;
        for (int w = 0; w < kMegaWarps; ++w) v += wred[w * NB * 32 + b * 32 + lane];
        const int n = rg * 32 + lane;
        if (n < ph.n_valid) {
          if (a.logits) a.logits[(size_t)b * a.logits_stride + n] = v;
          if (argmax_better(v, n, best_v[b], best_i[b])) { best_v[b] = v; best_i[b] = n; }
        }
      }
    }
    __syncthreads();
  }
  if (warp == 0) {
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

template <int NB>
__global__ void __launch_bounds__(kMegaThreads, 1) mega_step_kernel(const MegaArgs a) {
  extern __shared__ __align__(16) float msmem[];
  __shared__ int abort_s;
  if (blockIdx.x == 0 && threadIdx.x < a.nb) {
    const int t = a.tok_idx ? a.tokens[a.tok_idx[threadIdx.x]] : a.tokens[threadIdx.x];
    if (t < 0 || t >= a.V) set_err(a.err, G4_DEV_BAD_TOKEN);
  }
  if (a.stamps && blockIdx.x == 0 && threadIdx.x == 0) a.stamps[0] = globaltimer_ns();
  for (int p = 0; p < a.n_phases; ++p) {
    const MegaPhase& ph = a.phases[p];
    switch (ph.type) {
      case PH_PMP:
      case PH_GEMV:
        if (ph.fmt == FMT_W4A16) mega_gemv<FMT_W4A16, NB>(a, ph, msmem);
        else mega_gemv<FMT_BF16, NB>(a, ph, msmem);
        break;
      case PH_PLE:
        mega_ple<NB>(a, ph, msmem);
        break;
      case PH_ATTN:
        switch (ph.attn_d) {
          case 64: mega_attn_d<64>(a, ph, reinterpret_cast<unsigned char*>(msmem)); break;
          case 128: mega_attn_d<128>(a, ph, reinterpret_cast<unsigned char*>(msmem)); break;
          case 256: mega_attn_d<256>(a, ph, reinterpret_cast<unsigned char*>(msmem)); break;
          default: mega_attn_d<512>(a, ph, reinterpret_cast<unsigned char*>(msmem)); break;
        }
        break;
      case PH_LMHEAD:
        mega_lmhead<NB>(a, ph, msmem);
        break;
      case PH_ARGMAX:
        mega_argmax<NB>(a, msmem);
        break;
    }
    if (p + 1 < a.n_phases && !grid_sync(a, (unsigned)p, &abort_s)) return;
    if (a.stamps && blockIdx.x == 0 && threadIdx.x == 0) a.stamps[p + 1] = globaltimer_ns();
  }
}

}  // namespace g4
