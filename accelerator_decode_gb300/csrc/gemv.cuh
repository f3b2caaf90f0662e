// Weight-only projections for small batches (GEMV): y[b, n] = sum_k W[n, k] x[b, k].
//
// Device weight layout ("lane = row" tiles).  Rows are grouped in blocks of 32 (one per
// lane); K is cut into 16-byte tiles per lane:
//   W4A16: tile = one group of 32 int4 (16 B) of one row, offset-binary nibbles n = q + 8;
//          word m (0..3) of a tile holds k = 8m..8m+7 of the group with k = 8m+2j at bits
//          [4j, 4j+4) and k = 8m+2j+1 at bits [16+4j, 20+4j) (j = 0..3), so one mask+OR
//          turns a nibble pair into a bf16x2 (128+n_even, 128+n_odd).
//   bf16:  tile = 8 consecutive bf16 of one row.
//   qw[(rb * tiles_per_row + t) * 32 + lane]: a warp reads 512 contiguous bytes per tile.
//   W4A16 scales: sc[(rb * S + sg) * 32 + lane] = 8 bf16 (the 8 groups of supergroup sg).
// A "supergroup" is 8 tiles of a row (256 k for W4A16, 64 k for bf16).
//
// Dequantisation is bf16(q * s): the nibble becomes an exact bf16 q by one subtraction
// (bf16 128+n minus 136), then one bf16x2 multiply rounds q*s to nearest even, as
// dequantising to bf16 does ("One TPU chip, eight agents", Two optimizations that didn't
// work; "Gemma 4 E2B in Pure JAX on a Colab TPU", cell 1.2).  Accumulation is fp32 (packed
// fp32x2 FMA) with fp32 activations.
//
// Work: CTA = 4 warps on one row group (R row blocks) and one K slice; warps take different
// supergroups of the slice.  With one K slice, CTAs loop over row groups (persistent) and
// prefetch the next row group's weights before reducing the current one; with several, the
// last CTA of a row group sums the slices' partials in slice order (deterministic).
// Latency: the first weights are requested before griddepcontrol.wait (programmatic
// dependent launch), and the activation rows are staged with one wave of cp.async.
#pragma once
#include "common.cuh"

namespace g4 {

enum { FMT_BF16 = 0, FMT_W4A16 = 1 };
enum { PRO_PLAIN = 0, PRO_NORM = 1, PRO_RESID = 2, PRO_GEGLU = 3, PRO_PLEG = 4 };  // last two: staged GEMV only
enum { EPI_STORE = 0, EPI_GEGLU = 1, EPI_PLE = 2, EPI_ARGMAX = 3 };

constexpr int kGemvWarps = 4;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kMaxNB = 4;  // batch rows per GEMV launch

struct GemvArgs {
  const uint4* qw;
  const uint4* sc;
  int n_rb;       // 32-row blocks (padded)
  int n_valid;    // valid outputs (rows; for GEGLU: output features)
  int K;          // logical inner size (multiple of 32)
  int S;          // supergroups along K
  int tiles;      // tiles per row = 8 * S
  int nb;         // batch rows in this launch (<= kMaxNB)
  int ksplit;     // K slices (CTAs along K per row group)
  int sg_per_cta; // supergroups per slice
  // prologue
  int pro;
  const float* x_in;
  int x_stride;
  const float* r_in;
  int r_stride;
  int r_parts;        // > 1: r_in holds K-slice partial sums, part q at r_in + q * r_part_stride
  long r_part_stride;
  const __nv_bfloat16* g_r;
  float lambda;
  const __nv_bfloat16* g_a;
  float* x_out;
  float eps;
  int norm_n;     // length of the residual vector (== K for PRO_NORM / PRO_RESID)
  // epilogue
  float* y;
  int y_stride;
  const float* ple;
  int ple_stride;
  float* logits;   // EPI_ARGMAX: optional [nb, logits_stride]
  int logits_stride;
  float* am_val;   // EPI_ARGMAX partials [nb][gridDim.x]
  int* am_idx;
  int* next_ids;   // EPI_ARGMAX: [nb]
  // split-K scratch
  float* part;     // [ksplit][nb][n_rb * 32]
  unsigned* counters;
};

template <int FMT>
struct Fmt {
  static constexpr int SGK = FMT == FMT_W4A16 ? 256 : 64;  // k per supergroup
  static constexpr int TK = SGK / 8;                        // k per tile
};

// Shared-memory plan (floats), identical on host and device.
struct GemvSmem {
  int xs, red, stage, gath, total_floats;
};
__host__ __device__ inline GemvSmem gemv_smem_plan(int NB, int R, int kc, int pro, int n, int ksplit) {
  GemvSmem p;
  const int nv = R * NB * 32;
  int red = (kGemvWarps + 1) * nv;
  if (red < 32 * NB) red = 32 * NB;
  p.xs = 0;
  p.red = NB * kc;
  p.stage = p.red + red;
  const int stage = pro == PRO_PLAIN ? 0 : 2 * NB * n + n;  // x rows, r rows, two bf16 gain vectors
  p.gath = p.stage + stage;
  p.total_floats = p.gath + (ksplit > 1 ? nv * ksplit : 0);
  return p;
}

// Accumulate one tile (one row, TK k values) into acc[b] for NB activation rows.
template <int FMT, int NB>
__device__ __forceinline__ void tile_fma(const uint4 wv, uint32_t s2, const float* xs, int xs_stride,
                                         float2 (&acc)[NB]) {
  const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
  if constexpr (FMT == FMT_W4A16) {
    const __nv_bfloat162 bias = __floats2bfloat162_rn(136.f, 136.f);
    const __nv_bfloat162 sc = as_bf162(s2);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float4 xa[NB], xb[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        xa[b] = *reinterpret_cast<const float4*>(xs + b * xs_stride + 8 * m);
        xb[b] = *reinterpret_cast<const float4*>(xs + b * xs_stride + 8 * m + 4);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t u = ((w[m] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
        __nv_bfloat162 q = __hsub2(as_bf162(u), bias);
        uint32_t p = as_u32(__hmul2(q, sc));
        float2 wf = make_float2(bf16_lo(p), bf16_hi(p));
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float2 xv = j == 0 ? make_float2(xa[b].x, xa[b].y)
                    : j == 1 ? make_float2(xa[b].z, xa[b].w)
                    : j == 2 ? make_float2(xb[b].x, xb[b].y)
                             : make_float2(xb[b].z, xb[b].w);
          acc[b] = __ffma2_rn(wf, xv, acc[b]);
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
    for (int m = 0; m < 4; ++m) {
      float2 wf = make_float2(bf16_lo(w[m]), bf16_hi(w[m]));
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float2 xv = m == 0 ? make_float2(xa[b].x, xa[b].y)
                  : m == 1 ? make_float2(xa[b].z, xa[b].w)
                  : m == 2 ? make_float2(xb[b].x, xb[b].y)
                           : make_float2(xb[b].z, xb[b].w);
        acc[b] = __ffma2_rn(wf, xv, acc[b]);
      }
    }
  }
}

// Prologue: stage the activation chunk [k0, k0 + kc) of NB rows into xs (fp32), zero-padded
// beyond k1 and beyond nb.  PRO_NORM / PRO_RESID first stage whole rows (one cp.async wave),
// then reduce from shared memory.
template <int NB>
__device__ __forceinline__ void gemv_prologue(const GemvArgs& a, float* smem, const GemvSmem& L, int kc, int k0,
                                              int k1) {
  const int tid = threadIdx.x, nt = blockDim.x;
  float* xs = smem + L.xs;
  float* red = smem + L.red;
  if (a.pro == PRO_PLAIN) {
    const int c4 = kc / 4;
    for (int i = tid; i < NB * c4; i += nt) {
      const int b = i / c4, c = i - b * c4, k = k0 + 4 * c;
      const bool ok = b < a.nb && k < k1;
      cp_async16(xs + b * kc + 4 * c, ok ? a.x_in + (size_t)b * a.x_stride + k : a.x_in, ok);
    }
    cp_async_wait_all();
    __syncthreads();
    return;
  }
  const int n = a.norm_n;
  float* xin = smem + L.stage;
  float* rin = xin + NB * n;
  __nv_bfloat16* gr = reinterpret_cast<__nv_bfloat16*>(rin + NB * n);
  __nv_bfloat16* ga = gr + n;
  const bool resid = a.pro == PRO_RESID;
  const int c4 = n / 4;
  const bool r_split = resid && a.r_parts > 1;
  for (int i = tid; i < NB * c4; i += nt) {
    const int b = i / c4, c = i - b * c4;
    const bool ok = b < a.nb;
    cp_async16(xin + b * n + 4 * c, ok ? a.x_in + (size_t)b * a.x_stride + 4 * c : a.x_in, ok);
    if (resid && !r_split) cp_async16(rin + b * n + 4 * c, ok ? a.r_in + (size_t)b * a.r_stride + 4 * c : a.r_in, ok);
    if (r_split) {  // the branch's K-slice parts, added in part order
      float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
      if (ok) {
        const float4* src = reinterpret_cast<const float4*>(a.r_in + (size_t)b * a.r_stride) + c;
        r = __ldcg(src);
        for (int q = 1; q < a.r_parts; ++q) {
          const float4 v = __ldcg(src + q * a.r_part_stride / 4);
          r.x += v.x;
          r.y += v.y;
          r.z += v.z;
          r.w += v.w;
        }
      }
      *reinterpret_cast<float4*>(rin + b * n + 4 * c) = r;
    }
  }
  for (int i = tid; i < n / 8; i += nt) {
    if (resid) cp_async16(gr + 8 * i, a.g_r + 8 * i, true);
    if (a.g_a) cp_async16(ga + 8 * i, a.g_a + 8 * i, true);
  }
  cp_async_wait_all();
  __syncthreads();
  if (resid) {
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ss[b] = 0.f;
      for (int k = tid; k < n; k += nt) ss[b] += rin[b * n + k] * rin[b * n + k];
    }
    block_sum<NB>(ss, red);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float rd = rms_denom(ss[b], n, a.eps);
      for (int k = tid; k < n; k += nt)
        xin[b * n + k] = (xin[b * n + k] + (rin[b * n + k] / rd) * bf16f(gr[k])) * a.lambda;
    }
    __syncthreads();
    if (blockIdx.x == 0) {
      for (int i = tid; i < a.nb * c4; i += nt) {
        const int b = i / c4, c = i - b * c4;
        *reinterpret_cast<float4*>(a.x_out + (size_t)b * a.x_stride + 4 * c) =
            *reinterpret_cast<const float4*>(xin + b * n + 4 * c);
      }
    }
  }
  float ad[NB];
  if (a.g_a != nullptr) {
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ad[b] = 0.f;
      for (int k = tid; k < n; k += nt) ad[b] += xin[b * n + k] * xin[b * n + k];
    }
    block_sum<NB>(ad, red);
#pragma unroll
    for (int b = 0; b < NB; ++b) ad[b] = rms_denom(ad[b], n, a.eps);
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    for (int k = k0 + tid; k < k0 + kc; k += nt) {
      float v = 0.f;
      if (b < a.nb && k < k1) {
        v = xin[b * n + k];
        if (a.g_a != nullptr) v = (v / ad[b]) * bf16f(ga[k]);
      }
      xs[b * kc + (k - k0)] = v;
    }
  }
  __syncthreads();
}

template <int FMT, int R, int NB, int EPI>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvArgs a) {
  using F = Fmt<FMT>;
  extern __shared__ __align__(16) float smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x % a.ksplit;
  const int rg_step = gridDim.x / a.ksplit;
  const int n_rg = a.n_rb / R;
  const int sg0 = ks * a.sg_per_cta;
  const int sg1 = min(a.S, sg0 + a.sg_per_cta);
  const int kc = a.sg_per_cta * F::SGK;
  const int k0 = sg0 * F::SGK;
  const int k1 = min(a.K, sg1 * F::SGK);
  const GemvSmem L = gemv_smem_plan(NB, R, kc, a.pro, a.norm_n, a.ksplit);
  const int rows_total = a.n_rb * 32;
  // Warp w takes tiles i = w, w + 4, ... of the CTA's K slice (tile i: supergroup sg0 + i / 8,
  // tile i % 8), so every warp has work whatever the slice's supergroup count.  Weights move
  // through a two-group register pipeline of kGrp tiles; the first group is loaded before
  // waiting on the previous kernel, the next row group's first group before the reduction.
  constexpr int kGrp = 8 / R;  // 8 tiles (R = 1) or 4 tile pairs (R = 2) per group
  const int nT = (sg1 - sg0) * 8;
  const int nj = nT > warp ? (nT - warp + kGemvWarps - 1) / kGemvWarps : 0;  // tiles of this warp
  const int ng = (nj + kGrp - 1) / kGrp;

  uint4 wb0[kGrp][R], wb1[kGrp][R];
  uint32_t sw0[kGrp][R], sw1[kGrp][R];
  auto load_grp = [&](uint4 (&wb)[kGrp][R], uint32_t (&sw)[kGrp][R], int rg_, int gi) {
#pragma unroll
    for (int g = 0; g < kGrp; ++g) {
      const int i = warp + kGemvWarps * (gi * kGrp + g);
      if (i < nT) {
        const int s = sg0 + (i >> 3), t = i & 7;
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int rb = rg_ * R + r;
          wb[g][r] = __ldg(a.qw + ((size_t)rb * a.tiles + (size_t)s * 8 + t) * 32 + lane);
          if constexpr (FMT == FMT_W4A16)
            sw[g][r] = __ldg(reinterpret_cast<const uint32_t*>(a.sc + ((size_t)rb * a.S + s) * 32 + lane) + (t >> 1));
        }
      }
    }
  };
  int rg = blockIdx.x / a.ksplit;
  if (rg < n_rg && ng > 0) load_grp(wb0, sw0, rg, 0);  // weights never depend on activations
  pdl_wait();
  pdl_trigger();
  gemv_prologue<NB>(a, smem, L, kc, k0, k1);

  float* xs = smem + L.xs;
  float* red = smem + L.red;
  constexpr int NV = R * NB * 32;
  float* fin = red + kGemvWarps * NV;
  float best_v[NB];
  int best_i[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) { best_v[b] = __int_as_float(0x7fc00000); best_i[b] = 0x7fffffff; }

  for (; rg < n_rg; rg += rg_step) {
    float2 acc[R][NB];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) acc[r][b] = make_float2(0.f, 0.f);
    auto compute_grp = [&](const uint4 (&wb)[kGrp][R], const uint32_t (&sw)[kGrp][R], int gi) {
#pragma unroll
      for (int g = 0; g < kGrp; ++g) {
        const int i = warp + kGemvWarps * (gi * kGrp + g);
        if (i < nT) {
          const int t = i & 7;
          const float* xt = xs + (i >> 3) * F::SGK + t * F::TK;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            uint32_t s2 = 0;
            if constexpr (FMT == FMT_W4A16) {
              const uint32_t hh = (t & 1) ? (sw[g][r] >> 16) : (sw[g][r] & 0xFFFFu);
              s2 = hh | (hh << 16);
            }
            tile_fma<FMT, NB>(wb[g][r], s2, xt, kc, acc[r]);
          }
        }
      }
    };
    for (int gi = 0; gi < ng; ++gi) {
      if ((gi & 1) == 0) {
        if (gi + 1 < ng) load_grp(wb1, sw1, rg, gi + 1);
        compute_grp(wb0, sw0, gi);
      } else {
        if (gi + 1 < ng) load_grp(wb0, sw0, rg, gi + 1);
        compute_grp(wb1, sw1, gi);
      }
    }
    if (rg + rg_step < n_rg && ng > 0) load_grp(wb0, sw0, rg + rg_step, 0);  // next row group

    // cross-warp reduction in fixed warp order
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int b = 0; b < NB; ++b) red[warp * NV + (r * NB + b) * 32 + lane] = acc[r][b].x + acc[r][b].y;
    __syncthreads();
    for (int i = threadIdx.x; i < NV; i += blockDim.x) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kGemvWarps; ++w) s += red[w * NV + i];
      fin[i] = s;
    }
    __syncthreads();

    if (a.ksplit > 1) {  // one row group per CTA here (grid = n_rg * ksplit)
      for (int i = threadIdx.x; i < NV; i += blockDim.x) {
        const int b = (i / 32) % NB, r = i / (32 * NB), l = i % 32;
        if (b < a.nb) a.part[((size_t)ks * a.nb + b) * rows_total + (rg * R + r) * 32 + l] = fin[i];
      }
      __threadfence();
      __syncthreads();
      __shared__ int is_last;
      if (threadIdx.x == 0) is_last = atomicAdd(&a.counters[rg], 1u) == (unsigned)a.ksplit - 1;
      __syncthreads();
      if (!is_last) return;
      __threadfence();
      float* gath = smem + L.gath;  // [ksplit][NV]
      for (int i = threadIdx.x; i < NV * a.ksplit; i += blockDim.x) {
        const int q = i / NV, v = i - q * NV;
        const int b = (v / 32) % NB, r = v / (32 * NB), l = v % 32;
        gath[i] = b < a.nb ? ldcg(a.part + ((size_t)q * a.nb + b) * rows_total + (rg * R + r) * 32 + l) : 0.f;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < NV; i += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < a.ksplit; ++q) s += gath[q * NV + i];
        fin[i] = s;
      }
      if (threadIdx.x == 0) a.counters[rg] = 0u;
      __syncthreads();
    }

    if (warp == 0) {
      for (int b = 0; b < a.nb; ++b) {
        if constexpr (EPI == EPI_ARGMAX) {
          const int n = rg * 32 + lane;
          if (n < a.n_valid) {
            const float v = fin[b * 32 + lane];
            if (a.logits) a.logits[(size_t)b * a.logits_stride + n] = v;
            if (argmax_better(v, n, best_v[b], best_i[b])) { best_v[b] = v; best_i[b] = n; }
          }
        } else if constexpr (EPI == EPI_GEGLU) {
          const int n = rg * 32 + lane;  // R == 2: block 0 = gate rows, block 1 = up rows
          if (n < a.n_valid) {
            const float g = fin[(0 * NB + b) * 32 + lane], u = fin[(1 * NB + b) * 32 + lane];
            a.y[(size_t)b * a.y_stride + n] = gelu_tanh(g) * u;
          }
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int n = (rg * R + r) * 32 + lane;
            if (n >= a.n_valid) continue;
            float v = fin[(r * NB + b) * 32 + lane];
            if constexpr (EPI == EPI_PLE) v = gelu_tanh(v) * a.ple[(size_t)b * a.ple_stride + n];
            a.y[(size_t)b * a.y_stride + n] = v;
          }
        }
      }
    }
    __syncthreads();  // red/fin reuse by the next row group
  }

  if constexpr (EPI == EPI_ARGMAX) {
    // CTA partial (warp 0 holds the running bests), then the last CTA reduces all partials.
    __shared__ int is_last_am;
    if (warp == 0) {
      for (int b = 0; b < a.nb; ++b) {
        float v = best_v[b];
        int i = best_i[b];
        warp_argmax(v, i);
        if (lane == 0) {
          a.am_val[b * gridDim.x + blockIdx.x] = v;
          a.am_idx[b * gridDim.x + blockIdx.x] = i;
        }
      }
    }
    __threadfence();
    __syncthreads();
    unsigned* cnt = a.counters + n_rg;  // one past the per-row-group counters
    if (threadIdx.x == 0) is_last_am = atomicAdd(cnt, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last_am) return;
    __threadfence();
    __shared__ float rv[kGemvWarps];
    __shared__ int ri[kGemvWarps];
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
        for (int w = 1; w < kGemvWarps; ++w)
          if (argmax_better(rv[w], ri[w], rv[0], ri[0])) { rv[0] = rv[w]; ri[0] = ri[w]; }
        a.next_ids[b] = ri[0] == 0x7fffffff ? 0 : ri[0];
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) *cnt = 0u;
  }
}

}  // namespace g4
