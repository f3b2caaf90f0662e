// Staged weight-only projection for 1-4 activation rows: y[b, n] = sum_k W[n, k] x[b, k],
// on the GEMV tile layout of gemv.cuh (lane = row, 16-byte tiles, supergroups of 8 tiles).
//
// A decode step is a chain of dependent projections, each too small to keep HBM busy on its
// own, so the weights move ahead of the dependency: every CTA has a producer warp that
// streams its weight tiles into a shared-memory ring with bulk copies (cp.async.bulk,
// mbarrier completion) from the moment the CTA is resident -- under programmatic dependent
// launch that is while the previous kernel still computes -- and only the eight compute warps
// wait for the previous kernel (griddepcontrol.wait) before staging the activation rows with
// one wave of cp.async.  Norm gains are weights too: they are staged before the wait.
//
// Work.  K is cut into C slices of spc supergroups; CTA i owns slice i % C for the whole
// launch, and its producer takes row groups (R row blocks of 32 rows) one at a time from a
// counter of that slice (atomicAdd), as ring space frees.  A CTA that became resident late,
// or shares its SM with another CTA of the same launch, simply takes fewer row groups, so the
// split follows the speed each CTA actually gets.  The last CTA of a slice to finish taking
// resets the slice's counters for the next launch.  No sum crosses CTAs: slice c writes its
// raw partial sums to y + c * y_part_stride, and the kernel that reads them adds the C parts in
// slice order (deterministic) as it stages them, together with what an epilogue would apply
// (the GeGLU or per-layer-input gate of PRO_GEGLU / PRO_PLEG below, the residual update and
// norms of PRO_RESID, the q/k/v split in attention).
// Dequantisation and accumulation are those of the GEMV (tile_fma): bf16(q * s) weights,
// fp32 activations and sums.  Every wait is bounded; on expiry the CTA sets the device error
// word, stops, and waits (bounded) for the copies it issued before it exits.
//
// EPI_ARGMAX (the vocabulary projection and greedy choice, one K slice): a CTA takes as many
// row groups as its speed allows, so their sums cannot all stay in shared memory.  They go to
// a ring of `ru` unit slots instead; the warp that finishes a row group last (a shared-memory
// counter per slot) adds the eight warps' sums in warp order, writes the logits (if asked
// for) and keeps a running best per lane.  A slot is reused `ru` row groups later, which no
// warp reaches before that reduction is over (the ring of weights keeps the warps within
// `slots` items of one another, and ru * items per row group > slots + items per row group).
// The CTA's best goes to am_val / am_idx, and the last CTA to finish picks the winner
// (lowest index on ties, NaN never wins) into next_ids.
#pragma once
#include "common.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"

namespace g4 {

constexpr int kSgWarps = 8;                      // compute warps
constexpr int kSgThreads = (kSgWarps + 1) * 32;  // + the producer warp
constexpr int kSgMaxSlots = 16;
constexpr int kSgMaxUnits = 32;                  // row groups one CTA may take
constexpr int kSgMaxCsg = 4;                     // supergroups per ring item and row block
constexpr int kSgMaxRegs = 96;                   // registers per thread (launch padding relies on it)
constexpr int kSgMaxParts = 4;                   // K slices of one launch (and parts of an input)
constexpr unsigned long long kSgTimeoutNs = 1000000000ull;  // 1 s

struct GemvSArgs {
  const uint4* qw;
  const uint4* sc;
  int n_rb, S, tiles, K, n_valid;
  // partition (see the plan in g4.cu)
  int C;           // K slices; CTA i owns slice i % C
  int spc;         // supergroups per slice
  int csg;         // supergroups per ring item and row block (<= kSgMaxCsg)
  int slots;       // ring slots
  int slot_bytes;  // bytes per slot (multiple of 128)
  int cap;         // row groups one CTA may take (<= kSgMaxUnits)
  unsigned* grab;  // [C] row-group counters; zero before the launch, left zero after it
  unsigned* done;  // [C] CTAs of the slice that stopped taking
  int nb;          // activation rows (<= NB)
  // prologue (as GemvArgs, plus PRO_GEGLU / PRO_PLEG); the residual branch r and the
  // PRO_GEGLU / PRO_PLEG sources may come as K-slice parts to be added in part order
  int pro;
  const float* x_in;
  int x_stride;
  int x_parts;
  long x_part_stride;
  const float* r_in;
  int r_stride;
  int r_parts;
  long r_part_stride;
  const __nv_bfloat16* g_r;
  float lambda;
  const __nv_bfloat16* g_a;
  float* x_out;
  float eps;
  int norm_n;
  // output: slice c of row n of batch row b at y[c * y_part_stride + b * y_stride + n]
  float* y;
  int y_stride;
  long y_part_stride;
  const float* ple;  // PRO_PLEG: multipliers [nb][ple_stride]
  int ple_stride;
  int* err;
  // units whose sums shared memory holds: cap, or (EPI_ARGMAX) the ring of unit slots
  int ru;
  int am;          // 1: EPI_ARGMAX layout (per-slot counters in shared memory)
  float* am_val;   // EPI_ARGMAX: per-CTA bests [nb][grid]
  int* am_idx;
  unsigned* am_cnt;  // CTAs done; zero before the launch, left zero after it
  int* next_ids;     // [nb]
};

// Shared-memory plan (bytes from a 128-aligned base), identical on host and device.
//   ring | barriers, slot tags, unit rows, flags, (EPI_ARGMAX) slot counters | xs [NB][kc] |
//   stage (x rows, r rows, two gain vectors) | red [ru][warps][NV] | norm scratch [32][4 NB]
struct SgSmem {
  int bars, tags, units, xs, stage, red, nred, total;
};
__host__ __device__ inline SgSmem sg_smem_plan(int NB, int R, int sgk, const GemvSArgs& a) {
  SgSmem p;
  const int nv = R * NB * 32;
  int o = a.slots * a.slot_bytes;
  p.bars = o;
  o += (2 * a.slots + 1) * 8;  // full, empty, done
  p.tags = o;
  o += a.slots * 4;            // unit of each slot's item (-1: no more)
  p.units = o;
  o += kSgMaxUnits * 4 + 16;   // row group of each unit; abort, fail and last-CTA flags
  if (a.am) o += kSgMaxUnits * 4;  // warps done with each unit slot
  o = (o + 15) & ~15;
  p.xs = o;
  o += NB * a.spc * sgk * 4;
  p.stage = o;
  if (a.pro != PRO_PLAIN) o += (2 * NB * a.norm_n + a.norm_n) * 4;
  p.red = o;
  o += a.ru * kSgWarps * nv * 4;
  p.nred = o;
  o += 32 * 4 * NB * 4;
  p.total = o;
  return p;
}

__device__ __forceinline__ unsigned long long sg_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t sg_su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool sg_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(sg_su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait.  With abort_s != nullptr it also gives up once another role aborted.
__device__ __forceinline__ bool sg_wait(uint64_t* b, uint32_t parity, volatile int* abort_s) {
  unsigned long long t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (sg_try(b, parity)) return true;
    if ((i & 255u) == 255u) {
      if (abort_s && *abort_s) return false;
      const unsigned long long now = sg_now();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kSgTimeoutNs) return false;
    }
  }
}
__device__ __forceinline__ void sg_csync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kSgWarps * 32) : "memory"); }

// Sums of M values over the 256 compute threads (one barrier); `red` holds 32 * M floats.
template <int M>
__device__ __forceinline__ void sg_sum(float (&v)[M], float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int i = 0; i < M; ++i) v[i] = warp_sum(v[i]);
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < M; ++i) red[i * 32 + warp] = v[i];
  }
  sg_csync();
#pragma unroll
  for (int i = 0; i < M; ++i) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kSgWarps; ++w) s += red[i * 32 + w];
    v[i] = s;
  }
}

// Gains of the prologue (weights: staged before the dependency wait).
__device__ __forceinline__ void sg_stage_gains(const GemvSArgs& a, float* stage, int NB) {
  if (a.pro == PRO_PLAIN) return;
  const int n = a.norm_n;
  __nv_bfloat16* gr = reinterpret_cast<__nv_bfloat16*>(stage + 2 * NB * n);
  __nv_bfloat16* ga = gr + n;
  for (int i = threadIdx.x; i < n / 8; i += kSgWarps * 32) {
    if (a.pro == PRO_RESID) cp_async16(gr + 8 * i, a.g_r + 8 * i, true);
    if (a.g_a) cp_async16(ga + 8 * i, a.g_a + 8 * i, true);
  }
}

// Inputs that are a function of another projection's raw sums, over the K slice [k0, k1):
//   PRO_GEGLU: x[f] = gelu_tanh(g[f]) u[f], with g and u the gate and up rows of a tiled
//              [gate block j | up block j] matrix (row of gate f: 64 (f / 32) + f % 32, up: +32);
//   PRO_PLEG:  x[p] = gelu_tanh(g[p]) ple[p].
// All parts' loads are in flight together; they are added in part order.
template <int NB>
__device__ __forceinline__ void sg_gated_input(const GemvSArgs& a, float* xs, int kc, int k0, int k1) {
  const int tid = threadIdx.x, nt = kSgWarps * 32;
  const int c4 = kc / 4;
  const bool geglu = a.pro == PRO_GEGLU;
  // two chunks of four values per thread and pass: all their loads first
  for (int i0 = tid; i0 < NB * c4; i0 += 2 * nt) {
    float4 g[2][kSgMaxParts], u[2][kSgMaxParts], m[2];
    bool ok[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = i0 + h * nt, b = i / c4, c = i - b * c4, f = k0 + 4 * c;
      ok[h] = i < NB * c4 && b < a.nb && f < k1;
      if (!ok[h]) continue;
      const size_t rg_ = geglu ? (size_t)((f >> 5) << 6) + (f & 31) : (size_t)f;
      const float* base = a.x_in + (size_t)b * a.x_stride + rg_;
#pragma unroll
      for (int q = 0; q < kSgMaxParts; ++q) {
        if (q < a.x_parts) {
          g[h][q] = __ldcg(reinterpret_cast<const float4*>(base + q * a.x_part_stride));
          if (geglu) u[h][q] = __ldcg(reinterpret_cast<const float4*>(base + q * a.x_part_stride + 32));
        }
      }
      if (!geglu) m[h] = __ldcg(reinterpret_cast<const float4*>(a.ple + (size_t)b * a.ple_stride + f));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = i0 + h * nt, b = i / c4, c = i - b * c4;
      if (i >= NB * c4) continue;
      float4 out = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok[h]) {
        float4 gs = g[h][0], us = geglu ? u[h][0] : m[h];
#pragma unroll
        for (int q = 1; q < kSgMaxParts; ++q) {
          if (q < a.x_parts) {
            gs.x += g[h][q].x; gs.y += g[h][q].y; gs.z += g[h][q].z; gs.w += g[h][q].w;
            if (geglu) { us.x += u[h][q].x; us.y += u[h][q].y; us.z += u[h][q].z; us.w += u[h][q].w; }
          }
        }
        out = make_float4(gelu_tanh(gs.x) * us.x, gelu_tanh(gs.y) * us.y, gelu_tanh(gs.z) * us.z,
                          gelu_tanh(gs.w) * us.w);
      }
      *reinterpret_cast<float4*>(xs + b * kc + 4 * c) = out;
    }
  }
  sg_csync();
}

// Activation prologue on the compute warps (after the dependency wait): the K slice
// [k0, k0 + kc) of NB rows into xs (zero beyond k1 and beyond nb).  PRO_NORM / PRO_RESID stage
// whole rows first (one cp.async wave; the residual branch's parts land side by side in the
// x-row area and are added in part order), then one pass takes all the sums the norms need,
// one barrier adds them over the warps, and one pass writes the slice (and, in the grid's
// first CTA, the updated residual).  With x' = lambda (x + r g_r / d_r), d_r = sqrt(mean r^2 +
// eps), the second norm's sum of squares is
//   sum x'^2 = lambda^2 (sum x^2 + (2 / d_r) sum x r g_r + (1 / d_r^2) sum r^2 g_r^2),
// so it needs no second pass.
template <int NB>
__device__ __forceinline__ void sg_prologue(const GemvSArgs& a, float* xs, float* stage, float* nred, int kc, int k0,
                                            int k1) {
  const int tid = threadIdx.x, nt = kSgWarps * 32;
  if (a.pro == PRO_GEGLU || a.pro == PRO_PLEG) {
    sg_gated_input<NB>(a, xs, kc, k0, k1);
    return;
  }
  if (a.pro == PRO_PLAIN) {
    const int c4 = kc / 4;
    for (int i = tid; i < NB * c4; i += nt) {
      const int b = i / c4, c = i - b * c4, k = k0 + 4 * c;
      const bool ok = b < a.nb && k < k1;
      cp_async16(xs + b * kc + 4 * c, ok ? a.x_in + (size_t)b * a.x_stride + k : a.x_in, ok);
    }
    cp_async_wait_all();
    sg_csync();
    return;
  }
  const int n = a.norm_n;
  float* xin = stage;
  float* rin = xin + NB * n;
  const __nv_bfloat16* gr = reinterpret_cast<const __nv_bfloat16*>(rin + NB * n);
  const __nv_bfloat16* ga = gr + n;
  const bool resid = a.pro == PRO_RESID;
  const bool norm = a.g_a != nullptr;
  const int c4 = n / 4;
  const int parts = resid ? a.r_parts : 0;
  for (int i = tid; i < NB * c4; i += nt) {
    const int b = i / c4, c = i - b * c4;
    const bool ok = b < a.nb;
    cp_async16(xin + b * n + 4 * c, ok ? a.x_in + (size_t)b * a.x_stride + 4 * c : a.x_in, ok);
    if (parts == 1) cp_async16(rin + b * n + 4 * c, ok ? a.r_in + (size_t)b * a.r_stride + 4 * c : a.r_in, ok);
  }
  if (parts > 1) {
    // r in slices: two chunks per thread and pass, every part's loads in flight at once, added
    // in part order
    for (int i0 = tid; i0 < NB * c4; i0 += 2 * nt) {
      float4 v[2][kSgMaxParts];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = i0 + h * nt, b = i / c4, c = i - b * c4;
#pragma unroll
        for (int q = 0; q < kSgMaxParts; ++q)
          if (i < NB * c4 && q < parts && b < a.nb)
            v[h][q] = __ldcg(reinterpret_cast<const float4*>(a.r_in + q * a.r_part_stride + (size_t)b * a.r_stride) + c);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = i0 + h * nt, b = i / c4, c = i - b * c4;
        if (i >= NB * c4) continue;
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        if (b < a.nb) {
          r = v[h][0];
#pragma unroll
          for (int q = 1; q < kSgMaxParts; ++q) {
            if (q < parts) {
              r.x += v[h][q].x;
              r.y += v[h][q].y;
              r.z += v[h][q].z;
              r.w += v[h][q].w;
            }
          }
        }
        *reinterpret_cast<float4*>(rin + b * n + 4 * c) = r;
      }
    }
  }
  cp_async_wait_all();
  sg_csync();
  // per row: sum x^2, sum r^2, sum x r g_r, sum r^2 g_r^2
  float t[4 * NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    float sx = 0.f, sr = 0.f, sxr = 0.f, srr = 0.f;
    for (int k = tid; k < n; k += nt) {
      const float x = xin[b * n + k];
      sx += x * x;
      if (resid) {
        const float r = rin[b * n + k], rg = r * bf16f(gr[k]);
        sr += r * r;
        sxr += x * rg;
        srr += rg * rg;
      }
    }
    t[4 * b] = sx;
    t[4 * b + 1] = sr;
    t[4 * b + 2] = sxr;
    t[4 * b + 3] = srr;
  }
  sg_sum<4 * NB>(t, nred);
  float inv_r[NB], inv_a[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    inv_r[b] = resid ? 1.0f / rms_denom(t[4 * b + 1], n, a.eps) : 0.f;
    float ss = t[4 * b];
    if (resid) ss = a.lambda * a.lambda * (ss + 2.0f * inv_r[b] * t[4 * b + 2] + inv_r[b] * inv_r[b] * t[4 * b + 3]);
    inv_a[b] = norm ? 1.0f / rms_denom(ss, n, a.eps) : 1.f;
  }
  const bool write_x = resid && blockIdx.x == 0;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (write_x && b < a.nb) {
      for (int c = tid; c < c4; c += nt) {
        float4 x = *reinterpret_cast<const float4*>(xin + b * n + 4 * c);
        const float4 r = *reinterpret_cast<const float4*>(rin + b * n + 4 * c);
        x.x = (x.x + r.x * inv_r[b] * bf16f(gr[4 * c])) * a.lambda;
        x.y = (x.y + r.y * inv_r[b] * bf16f(gr[4 * c + 1])) * a.lambda;
        x.z = (x.z + r.z * inv_r[b] * bf16f(gr[4 * c + 2])) * a.lambda;
        x.w = (x.w + r.w * inv_r[b] * bf16f(gr[4 * c + 3])) * a.lambda;
        *reinterpret_cast<float4*>(a.x_out + (size_t)b * a.x_stride + 4 * c) = x;
      }
    }
    for (int k = k0 + tid; k < k0 + kc; k += nt) {
      float v = 0.f;
      if (b < a.nb && k < k1) {
        v = xin[b * n + k];
        if (resid) v = (v + rin[b * n + k] * inv_r[b] * bf16f(gr[k])) * a.lambda;
        if (norm) v = v * inv_a[b] * bf16f(ga[k]);
      }
      xs[b * kc + (k - k0)] = v;
    }
  }
  sg_csync();
}

// One tile position (TK values of k) of R row blocks against NB activation rows; the
// activation values are read once for all R blocks.  Same arithmetic as tile_fma.
template <int FMT, int NB, int R>
__device__ __forceinline__ void tiles_fma(const uint4 (&wv)[R], const uint32_t (&s2)[R], const float* xs,
                                          int xs_stride, float2 (&acc)[R][NB]) {
  if constexpr (FMT == FMT_W4A16) {
    const __nv_bfloat162 bias = __floats2bfloat162_rn(136.f, 136.f);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float4 xa[NB], xb[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        xa[b] = *reinterpret_cast<const float4*>(xs + b * xs_stride + 8 * m);
        xb[b] = *reinterpret_cast<const float4*>(xs + b * xs_stride + 8 * m + 4);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t w = m == 0 ? wv[r].x : m == 1 ? wv[r].y : m == 2 ? wv[r].z : wv[r].w;
        const __nv_bfloat162 sc = as_bf162(s2[r]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t u = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
          const uint32_t p = as_u32(__hmul2(__hsub2(as_bf162(u), bias), sc));
          const float2 wf = make_float2(bf16_lo(p), bf16_hi(p));
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const float2 xv = j == 0 ? make_float2(xa[b].x, xa[b].y)
                            : j == 1 ? make_float2(xa[b].z, xa[b].w)
                            : j == 2 ? make_float2(xb[b].x, xb[b].y)
                                     : make_float2(xb[b].z, xb[b].w);
            acc[r][b] = __ffma2_rn(wf, xv, acc[r][b]);
          }
        }
      }
    }
  } else {
    float4 xa[NB], xb[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      xa[b] = *reinterpret_cast<const float4*>(xs + b * xs_stride);
      xb[b] = *reinterpret_cast<const float4*>(xs + b * xs_stride + 4);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t w[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 wf = make_float2(bf16_lo(w[m]), bf16_hi(w[m]));
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const float2 xv = m == 0 ? make_float2(xa[b].x, xa[b].y)
                          : m == 1 ? make_float2(xa[b].z, xa[b].w)
                          : m == 2 ? make_float2(xb[b].x, xb[b].y)
                                   : make_float2(xb[b].z, xb[b].w);
          acc[r][b] = __ffma2_rn(wf, xv, acc[r][b]);
        }
      }
    }
  }
}

// Launched with kSgThreads threads, or with more (padding warps that only hold registers until
// the CTA ends: see the launch code); registers capped so that the padding arithmetic holds.
template <int FMT, int R, int NB, int EPI>
__global__ void __maxnreg__(kSgMaxRegs) gemv_s_kernel(const GemvSArgs a) {
  using F = Fmt<FMT>;
  constexpr bool W4 = FMT == FMT_W4A16;
  constexpr int NV = R * NB * 32;
  constexpr uint32_t kSgW = 8 * 512;           // weight bytes of one supergroup of one row block
  constexpr uint32_t kSgS = W4 ? 512 : 0;      // its scale bytes
  extern __shared__ __align__(128) uint8_t sg_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sg_raw) + 127) & ~uintptr_t(127));
  const SgSmem L = sg_smem_plan(NB, R, F::SGK, a);
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* empty = full + a.slots;
  uint64_t* done = empty + a.slots;               // the compute warps have finished (producer drain)
  volatile int* tag = reinterpret_cast<volatile int*>(smem + L.tags);     // [slots] unit of the item
  volatile int* unit_rg = reinterpret_cast<volatile int*>(smem + L.units);  // [ru] row group of a unit slot
  volatile int* abort_s = unit_rg + kSgMaxUnits;  // tells the producer to stop
  volatile int* cfail = abort_s + 1;              // compute warps: written before a barrier, read after it
  volatile int* am_last = abort_s + 2;            // EPI_ARGMAX: this CTA finished last
  unsigned* ucnt = reinterpret_cast<unsigned*>(const_cast<int*>(abort_s + 4));  // EPI_ARGMAX: [ru]
  float* xs = reinterpret_cast<float*>(smem + L.xs);
  float* stage = reinterpret_cast<float*>(smem + L.stage);
  float* red = reinterpret_cast<float*>(smem + L.red);  // [cap][warps][NV]
  float* nred = reinterpret_cast<float*>(smem + L.nred);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x % a.C;                // this CTA's K slice
  const int n_rg = a.n_rb / R;
  const int sg0 = ks * a.spc;
  const int sg1 = min(a.S, sg0 + a.spc);
  const int nch = (max(0, sg1 - sg0) + a.csg - 1) / a.csg;  // ring items per row group
  const int kc = a.spc * F::SGK;
  const int k0 = sg0 * F::SGK;
  const int k1 = min(a.K, sg1 * F::SGK);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.slots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSgWarps);
    }
    mbar_init(done, 1);
    *abort_s = 0;
    *cfail = 0;
    if constexpr (EPI == EPI_ARGMAX)
      for (int i = 0; i < a.ru; ++i) ucnt[i] = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();

  if (warp > kSgWarps) {  // padding: stay resident until the compute warps are done
    if (lane == 0) sg_wait(done, 0, nullptr);
    return;
  }
  if (warp == kSgWarps) {
    // ---------------- producer: weights only (no dependency on the previous kernel)
    if (lane == 0) {
      int it = 0;
      bool dead = false;
      auto slot_free = [&](int s, int ph) {  // the consumers released the slot's previous item
        if (ph == 0) return true;
        if (sg_wait(&empty[s], (ph - 1) & 1, abort_s)) return true;
        if (!*abort_s) { set_err(a.err, G4_DEV_TIMEOUT); *abort_s = 1; }
        return false;
      };
      for (int u = 0; u < a.cap && !dead; ++u) {
        // take the next row group only once the ring has room for its first item
        if (!slot_free(it % a.slots, it / a.slots)) { dead = true; break; }
        const int rg = (int)atomicAdd(&a.grab[ks], 1u);
        if (rg >= n_rg) break;
        unit_rg[u % a.ru] = rg;
        for (int c = 0; c < nch; ++c, ++it) {
          const int s = it % a.slots, ph = it / a.slots;
          if (c > 0 && !slot_free(s, ph)) { dead = true; break; }
          const int cs0 = sg0 + c * a.csg;
          const int ncs = min(sg1, cs0 + a.csg) - cs0;
          uint8_t* dst = ring + (size_t)s * a.slot_bytes;
          tag[s] = u;
          mbar_expect_tx(&full[s], (uint32_t)(R * ncs * (kSgW + kSgS)));  // releases tag and unit_rg
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const size_t rb = (size_t)rg * R + r;
            bulk_g2s(dst + r * ncs * kSgW, a.qw + (rb * a.tiles + (size_t)cs0 * 8) * 32, ncs * kSgW, &full[s]);
            if constexpr (W4)
              bulk_g2s(dst + R * ncs * kSgW + r * ncs * kSgS, a.sc + (rb * a.S + cs0) * 32, ncs * kSgS, &full[s]);
          }
        }
      }
      // the slice's counters go back to zero once every CTA of the slice has stopped taking
      __threadfence();
      if (atomicAdd(&a.done[ks], 1u) == gridDim.x / a.C - 1) {
        atomicExch(&a.grab[ks], 0u);
        atomicExch(&a.done[ks], 0u);
      }
      // end mark for the consumers (an item without data)
      bool marked = false;
      if (!dead && slot_free(it % a.slots, it / a.slots)) {
        tag[it % a.slots] = -1;
        mbar_arrive(&full[it % a.slots]);
        marked = true;
      }
      // No copy may be in flight into this CTA's shared memory when it exits: wait for the last
      // item of every slot.  The end mark's slot held item it - slots, which the consumers had
      // released (so it had landed) before the mark went in; its barrier is a phase further on.
      for (int j = max(0, it - a.slots); j < it; ++j)
        if (!(marked && j == it - a.slots)) sg_wait(&full[j % a.slots], (j / a.slots) & 1, nullptr);
      sg_wait(done, 0, nullptr);
    }
    return;
  }

  // ---------------- compute warps
  struct DoneOnExit {  // lets the producer leave on every way out of the compute warps
    uint64_t* b;
    __device__ ~DoneOnExit() {
      if (threadIdx.x == 0) mbar_arrive(b);
    }
  } done_on_exit{done};
  sg_stage_gains(a, stage, NB);  // weights: before the dependency wait
  pdl_wait();
  pdl_trigger();
  sg_prologue<NB>(a, xs, stage, nred, kc, k0, k1);
  // A failed wait is recorded in cfail before the next barrier of the compute warps and acted
  // on after it, so every warp leaves at the same point (no warp is left at a barrier).
  int units = 0;
  bool ok = true;
  float2 acc[R][NB];
  float best_v[NB];  // EPI_ARGMAX: running best of this lane's rows
  int best_i[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) { best_v[b] = __int_as_float(0x7fc00000); best_i[b] = 0x7fffffff; }
  for (int it = 0; ok; ++it) {
    const int s = it % a.slots, ph = it / a.slots;
    if (!sg_wait(&full[s], ph & 1, nullptr)) {
      ok = false;
      if (lane == 0) { set_err(a.err, G4_DEV_TIMEOUT); *cfail = 1; *abort_s = 1; }
      break;
    }
    const int u = tag[s];
    if (u < 0) break;  // no more row groups
    const int c = it - u * nch;
    if (c == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[r][b] = make_float2(0.f, 0.f);
    }
    const int cs0 = sg0 + c * a.csg;
    const int ncs = min(sg1, cs0 + a.csg) - cs0;
    const uint8_t* src = ring + (size_t)s * a.slot_bytes;
    // this warp's tiles of the item: tile `warp` of supergroup j of each row block (j < ncs);
    // all loads first, then the arithmetic
    uint4 wv[kSgMaxCsg][R];
    uint32_t s2[kSgMaxCsg][R];
#pragma unroll
    for (int j = 0; j < kSgMaxCsg; ++j) {
      if (j < ncs) {
        const int i = warp + 8 * j;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          wv[j][r] = *reinterpret_cast<const uint4*>(src + ((size_t)(r * ncs * 8 + i) * 32 + lane) * 16);
          s2[j][r] = 0;
          if constexpr (W4) {
            const uint32_t sw = *reinterpret_cast<const uint32_t*>(src + R * ncs * kSgW + (r * ncs + j) * kSgS +
                                                                   lane * 16 + (warp >> 1) * 4);
            const uint32_t hh = (warp & 1) ? (sw >> 16) : (sw & 0xFFFFu);
            s2[j][r] = hh | (hh << 16);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kSgMaxCsg; ++j) {
      if (j < ncs) {
        const float* xt = xs + (cs0 - sg0 + j) * F::SGK + warp * F::TK;
        tiles_fma<FMT, NB, R>(wv[j], s2[j], xt, kc, acc);
      }
    }
    __syncwarp();
    if constexpr (EPI == EPI_ARGMAX) {
      // the unit's reduction comes before this warp releases the slot (see the header)
      if (c == nch - 1) {
        const int us = u % a.ru;
        float* rb = red + (size_t)us * kSgWarps * NV;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int b = 0; b < NB; ++b) rb[warp * NV + (r * NB + b) * 32 + lane] = acc[r][b].x + acc[r][b].y;
        __syncwarp();
        unsigned prev = 0;
        if (lane == 0) {
          __threadfence_block();
          prev = atomicAdd(&ucnt[us], 1u);
        }
        prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
        if (prev == (unsigned)kSgWarps - 1) {  // the other warps' sums are in
          __threadfence_block();
          const int rg = unit_rg[us];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int n = (rg * R + r) * 32 + lane;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              float v = 0.f;
#pragma unroll
              for (int w = 0; w < kSgWarps; ++w) v += rb[w * NV + (r * NB + b) * 32 + lane];
              if (n < a.n_valid && b < a.nb) {
                if (a.y) a.y[(size_t)b * a.y_stride + n] = v;
                if (argmax_better(v, n, best_v[b], best_i[b])) { best_v[b] = v; best_i[b] = n; }
              }
            }
          }
          __syncwarp();
          if (lane == 0) ucnt[us] = 0u;
        }
      }
    }
    if (lane == 0) mbar_arrive(&empty[s]);
    if (EPI != EPI_ARGMAX && c == nch - 1) {
      // this warp's sums of unit u (its own slot: no barrier between row groups)
      float* rb = red + (size_t)u * kSgWarps * NV;
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < NB; ++b) rb[warp * NV + (r * NB + b) * 32 + lane] = acc[r][b].x + acc[r][b].y;
      units = u + 1;
    }
  }
  sg_csync();
  if (*cfail) return;
  if constexpr (EPI == EPI_ARGMAX) {
    // the CTA's best per batch row, then the grid's (last CTA), in index order on ties
    float* av = nred;
    int* ai = reinterpret_cast<int*>(nred + NB * kSgWarps);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float v = best_v[b];
      int i = best_i[b];
      warp_argmax(v, i);
      if (lane == 0) { av[b * kSgWarps + warp] = v; ai[b * kSgWarps + warp] = i; }
    }
    sg_csync();
    if (threadIdx.x == 0) {
      for (int b = 0; b < a.nb; ++b) {
        float v = av[b * kSgWarps];
        int i = ai[b * kSgWarps];
        for (int w = 1; w < kSgWarps; ++w)
          if (argmax_better(av[b * kSgWarps + w], ai[b * kSgWarps + w], v, i)) { v = av[b * kSgWarps + w]; i = ai[b * kSgWarps + w]; }
        a.am_val[b * gridDim.x + blockIdx.x] = v;
        a.am_idx[b * gridDim.x + blockIdx.x] = i;
      }
      __threadfence();
      *am_last = atomicAdd(a.am_cnt, 1u) == gridDim.x - 1;
    }
    sg_csync();
    if (!*am_last) return;
    __threadfence();
    for (int b = 0; b < a.nb; ++b) {
      float v = __int_as_float(0x7fc00000);
      int i = 0x7fffffff;
      for (int cta = threadIdx.x; cta < (int)gridDim.x; cta += kSgWarps * 32) {
        const float cv = ldcg(a.am_val + b * gridDim.x + cta);
        const int ci = __ldcg(a.am_idx + b * gridDim.x + cta);
        if (argmax_better(cv, ci, v, i)) { v = cv; i = ci; }
      }
      warp_argmax(v, i);
      if (lane == 0) { av[warp] = v; ai[warp] = i; }
      sg_csync();
      if (threadIdx.x == 0) {
        for (int w = 1; w < kSgWarps; ++w)
          if (argmax_better(av[w], ai[w], av[0], ai[0])) { av[0] = av[w]; ai[0] = ai[w]; }
        a.next_ids[b] = ai[0] == 0x7fffffff ? 0 : ai[0];
      }
      sg_csync();
    }
    if (threadIdx.x == 0) *a.am_cnt = 0u;
    return;
  }
  // outputs: value v = (r * NB + b) * 32 + lane of unit u is row (rg * R + r) * 32 + lane of
  // batch row b, summed over the warps in warp order
  float* ys = a.y + (size_t)ks * a.y_part_stride;
  for (int e = threadIdx.x; e < units * NV; e += kSgWarps * 32) {
    const int u = e / NV, v = e - u * NV;
    const int ln = v & 31, rbk = v >> 5, b = rbk % NB, r = rbk / NB;
    if (b >= a.nb) continue;
    const int rg = unit_rg[u];
    const float* rb = red + (size_t)u * kSgWarps * NV;
    auto sum_of = [&](int vv) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kSgWarps; ++w) sum += rb[w * NV + vv];
      return sum;
    };
    if constexpr (EPI == EPI_GEGLU) {
      if (r != 0) continue;
      const int n = rg * 32 + ln;  // R == 2: block 0 = gate rows, block 1 = up rows
      if (n < a.n_valid) ys[(size_t)b * a.y_stride + n] = gelu_tanh(sum_of(v)) * sum_of(v + NB * 32);
    } else {
      const int n = (rg * R + r) * 32 + ln;
      if (n >= a.n_valid) continue;
      float val = sum_of(v);
      if constexpr (EPI == EPI_PLE) val = gelu_tanh(val) * a.ple[(size_t)b * a.ple_stride + n];
      ys[(size_t)b * a.y_stride + n] = val;
    }
  }
}

}  // namespace g4
