// Decode attention with one KV head (MQA), split over keys (flash-decode).
//
// Per sequence b at position p, for the query heads of one head group:
//   q_h = RoPE(RMSNorm(q_raw_h) * g_q)                      (every layer)
//   owning layers: k = bf16(RoPE(RMSNorm(k_raw) * g_k)), v = bf16(v_raw) written in place
//   at cache row (slot, p) -- a sharing layer applies RoPE to its queries only and reads
//   its source layer's cache ("Porting Gemma 4 E2B to SGLang-JAX", Step 4; "One TPU chip,
//   eight agents", The engine: kv_share_map, static cache written in place).
//   keys j in [lo, p], lo = 0 (full) or max(0, p - W + 1) (sliding window W);
//   s_j = scale * q_h . K_j; o_h = sum_j softmax(s)_j V_j  (fp32, max-subtracted).
// The visible keys are cut into nsplit chunks (one CTA each) processed in tiles of 32 with
// an online softmax; the last CTA of a (sequence, head group) merges the chunks with their
// log-sum-exp weights.
#pragma once
#include "common.cuh"

namespace g4 {

constexpr int kAttnThreads = 128;
constexpr int kAttnTile = 32;

struct AttnArgs {
  const float* qkv;        // [nb][qkv_stride]: q heads, then k, v (owning layers)
  int qkv_stride;
  int nq;
  const __nv_bfloat16* g_q;
  const __nv_bfloat16* g_k;
  float eps;
  float scale;
  int window;              // 0 = full attention
  int own;                 // write K/V of this position
  __nv_bfloat16* kc;       // cache of the source layer [max_batch][t_max][D]
  __nv_bfloat16* vc;
  int t_max;
  int max_batch;
  const float* rope_cos;   // [t_max][D/2]
  const float* rope_sin;
  const int* slots;
  const int* positions;
  float* out;              // [nb][out_stride]
  int out_stride;
  int nsplit;
  float* ws_ml;            // [nb][nq][nsplit][2]
  float* ws_o;             // [nb][nq][nsplit][D]
  unsigned* counters;      // [nb][nq / HPC]
  int* err;
};

template <int D, int HPC>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  constexpr int PL = D / 32;        // q/k elements per lane (score phase)
  constexpr int PT = D >= kAttnThreads ? D / kAttnThreads : 1;  // output elements per thread
  static_assert(PL >= 2 && PL % 2 == 0, "head dim must be a multiple of 64");
  __shared__ __align__(16) float qs[HPC][D];
  __shared__ __align__(16) float knew[D];
  __shared__ __align__(16) float vnew[D];
  __shared__ float sc[HPC][kAttnTile];
  __shared__ float resc[HPC];
  __shared__ float red[32 * 2];
  const int split = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h0 = hg * HPC;
  const int n_hg = a.nq / HPC;

  int p = a.positions[b];
  const int slot = a.slots[b];
  bool bad = false;
  if (p < 0 || p >= a.t_max) { if (split == 0 && hg == 0 && tid == 0) set_err(a.err, G4_DEV_BAD_POSITION); bad = true; }
  if (slot < 0 || slot >= a.max_batch) { if (split == 0 && hg == 0 && tid == 0) set_err(a.err, G4_DEV_BAD_SLOT); bad = true; }
  if (bad) p = -1;
  const int lo = (p < 0) ? 0 : (a.window > 0 ? max(0, p - a.window + 1) : 0);
  const int nkeys = p - lo + 1;  // 0 when bad
  const int chunk = nkeys > 0 ? (nkeys + a.nsplit - 1) / a.nsplit : 0;
  const int j0 = lo + split * chunk;
  const int j1 = min(p + 1, j0 + chunk);
  const bool has_p = (p >= 0) && (j0 <= p) && (p < j1);

  // ---- q: per-head RMSNorm then RoPE at position p
  const float* qraw = a.qkv + (size_t)b * a.qkv_stride;
  if (j0 < j1) {
    for (int hh = warp; hh < HPC; hh += kAttnThreads / 32) {
      const float* src = qraw + (size_t)(h0 + hh) * D;
      float ss = 0.f;
      for (int e = lane; e < D; e += 32) ss += src[e] * src[e];
      ss = warp_sum(ss);
      const float den = rms_denom(ss, D, a.eps);
      for (int i = lane; i < D / 2; i += 32) {
        const float qa = (src[i] / den) * bf16f(a.g_q[i]);
        const float qb = (src[i + D / 2] / den) * bf16f(a.g_q[i + D / 2]);
        const float c = a.rope_cos[(size_t)p * (D / 2) + i], s = a.rope_sin[(size_t)p * (D / 2) + i];
        qs[hh][i] = qa * c - qb * s;
        qs[hh][i + D / 2] = qb * c + qa * s;
      }
    }
  }
  // ---- new K/V row of an owning layer (position p)
  if (a.own && has_p && warp == 0) {
    const float* kr = qraw + (size_t)a.nq * D;
    const float* vr = kr + D;
    float ss = 0.f;
    for (int e = lane; e < D; e += 32) ss += kr[e] * kr[e];
    ss = warp_sum(ss);
    const float den = rms_denom(ss, D, a.eps);
    __nv_bfloat16* kdst = a.kc + ((size_t)slot * a.t_max + p) * D;
    __nv_bfloat16* vdst = a.vc + ((size_t)slot * a.t_max + p) * D;
    for (int i = lane; i < D / 2; i += 32) {
      const float ka = (kr[i] / den) * bf16f(a.g_k[i]);
      const float kb = (kr[i + D / 2] / den) * bf16f(a.g_k[i + D / 2]);
      const float c = a.rope_cos[(size_t)p * (D / 2) + i], s = a.rope_sin[(size_t)p * (D / 2) + i];
      const __nv_bfloat16 k1 = __float2bfloat16_rn(ka * c - kb * s);
      const __nv_bfloat16 k2 = __float2bfloat16_rn(kb * c + ka * s);
      knew[i] = bf16f(k1);
      knew[i + D / 2] = bf16f(k2);
      if (hg == 0) { kdst[i] = k1; kdst[i + D / 2] = k2; }
    }
    for (int e = lane; e < D; e += 32) {
      const __nv_bfloat16 v1 = __float2bfloat16_rn(vr[e]);
      vnew[e] = bf16f(v1);
      if (hg == 0) vdst[e] = v1;
    }
  }
  __syncthreads();

  // ---- chunk: tiles of 32 keys, online softmax
  float m_run[HPC], l_run[HPC];
  float acc[HPC][PT];
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < PT; ++e) acc[h][e] = 0.f;
  }
  const __nv_bfloat16* kbase = a.kc + (size_t)(slot < 0 ? 0 : slot) * a.t_max * D;
  const __nv_bfloat16* vbase = a.vc + (size_t)(slot < 0 ? 0 : slot) * a.t_max * D;
  const bool use_new = a.own && has_p;

  for (int t0 = j0; t0 < j1; t0 += kAttnTile) {
    const int tn = min(kAttnTile, j1 - t0);
    // scores: warp per key, lanes over D
    for (int jj = warp; jj < kAttnTile; jj += kAttnThreads / 32) {
      const int j = t0 + jj;
      float kv[PL];
      if (jj < tn) {
        if (use_new && j == p) {
#pragma unroll
          for (int e = 0; e < PL; ++e) kv[e] = knew[lane * PL + e];
        } else {
          const __nv_bfloat16* kp = kbase + (size_t)j * D + lane * PL;
          if constexpr (PL % 8 == 0) {
#pragma unroll
            for (int c = 0; c < PL / 8; ++c) {
              const uint4 u = reinterpret_cast<const uint4*>(kp)[c];
              const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int m = 0; m < 4; ++m) { kv[c * 8 + 2 * m] = bf16_lo(w[m]); kv[c * 8 + 2 * m + 1] = bf16_hi(w[m]); }
            }
          } else {
#pragma unroll
            for (int c = 0; c < PL / 2; ++c) {
              const uint32_t w = reinterpret_cast<const uint32_t*>(kp)[c];
              kv[2 * c] = bf16_lo(w); kv[2 * c + 1] = bf16_hi(w);
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < HPC; ++h) {
        float d = 0.f;
        if (jj < tn) {
#pragma unroll
          for (int e = 0; e < PL; ++e) d += qs[h][lane * PL + e] * kv[e];
        }
        d = warp_sum(d);
        if (lane == 0) sc[h][jj] = (jj < tn) ? d * a.scale : -INFINITY;
      }
    }
    __syncthreads();
    // softmax statistics per head (warp per head)
    for (int h = warp; h < HPC; h += kAttnThreads / 32) {
      const float s = sc[h][lane];
      const float mt = warp_max(s);
      const float mn = fmaxf(m_run[h], mt);
      const float pj = (lane < tn) ? expf(s - mn) : 0.f;
      const float ls = warp_sum(pj);
      const float r = expf(m_run[h] - mn);  // 0 on the first tile
      sc[h][lane] = pj;
      if (lane == 0) resc[h] = r;
      m_run[h] = mn;
      l_run[h] = l_run[h] * r + ls;
    }
    __syncthreads();
    // P V: thread owns PT contiguous elements of each head's output
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      const float r = resc[h];
#pragma unroll
      for (int e = 0; e < PT; ++e) acc[h][e] *= r;
    }
    for (int jj = 0; jj < tn && tid * PT < D; ++jj) {
      const int j = t0 + jj;
      float vv[PT];
      if (use_new && j == p) {
#pragma unroll
        for (int e = 0; e < PT; ++e) vv[e] = vnew[tid * PT + e];
      } else {
        const __nv_bfloat16* vp = vbase + (size_t)j * D + tid * PT;
        if constexpr (PT == 1) {
          vv[0] = bf16f(vp[0]);
        } else if constexpr (PT == 2) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
          vv[0] = bf16_lo(w); vv[1] = bf16_hi(w);
        } else if constexpr (PT == 4) {
          const uint2 w = *reinterpret_cast<const uint2*>(vp);
          vv[0] = bf16_lo(w.x); vv[1] = bf16_hi(w.x); vv[2] = bf16_lo(w.y); vv[3] = bf16_hi(w.y);
        } else {
#pragma unroll
          for (int e = 0; e < PT; ++e) vv[e] = bf16f(vp[e]);
        }
      }
#pragma unroll
      for (int h = 0; h < HPC; ++h) {
        const float pj = sc[h][jj];
#pragma unroll
        for (int e = 0; e < PT; ++e) acc[h][e] += pj * vv[e];
      }
    }
    __syncthreads();
  }
  // m_run/l_run live in the stats warps; publish them through smem.
  __shared__ float m_sh[HPC], l_sh[HPC];
  for (int h = warp; h < HPC; h += kAttnThreads / 32)
    if (lane == 0) { m_sh[h] = m_run[h]; l_sh[h] = l_run[h]; }
  __syncthreads();

  float* outb = a.out + (size_t)b * a.out_stride;
  if (a.nsplit == 1) {
    if (tid * PT < D) {
#pragma unroll
      for (int h = 0; h < HPC; ++h) {
        const float L = l_sh[h];
#pragma unroll
        for (int e = 0; e < PT; ++e) outb[(h0 + h) * D + tid * PT + e] = L > 0.f ? acc[h][e] / L : 0.f;
      }
    }
    return;
  }
  // partial -> scratch
  const size_t base_ml = ((size_t)b * a.nq) * a.nsplit;
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    const size_t row = base_ml + (size_t)(h0 + h) * a.nsplit + split;
    if (tid == 0) { a.ws_ml[row * 2] = m_sh[h]; a.ws_ml[row * 2 + 1] = l_sh[h]; }
    if (tid * PT < D) {
#pragma unroll
      for (int e = 0; e < PT; ++e) a.ws_o[row * D + tid * PT + e] = acc[h][e];
    }
  }
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (tid == 0) is_last = atomicAdd(&a.counters[b * n_hg + hg], 1u) == (unsigned)a.nsplit - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int h = 0; h < HPC && tid * PT < D; ++h) {
    const size_t row0 = base_ml + (size_t)(h0 + h) * a.nsplit;
    float M = -INFINITY;
    for (int s = 0; s < a.nsplit; ++s) {
      const float l = ldcg(a.ws_ml + (row0 + s) * 2 + 1);
      if (l > 0.f) M = fmaxf(M, ldcg(a.ws_ml + (row0 + s) * 2));
    }
    float L = 0.f;
    float o[PT];
#pragma unroll
    for (int e = 0; e < PT; ++e) o[e] = 0.f;
    for (int s = 0; s < a.nsplit; ++s) {
      const float l = ldcg(a.ws_ml + (row0 + s) * 2 + 1);
      if (!(l > 0.f)) continue;
      const float w = expf(ldcg(a.ws_ml + (row0 + s) * 2) - M);
      L += w * l;
#pragma unroll
      for (int e = 0; e < PT; ++e) o[e] += w * ldcg(a.ws_o + (row0 + s) * D + tid * PT + e);
    }
#pragma unroll
    for (int e = 0; e < PT; ++e) outb[(h0 + h) * D + tid * PT + e] = L > 0.f ? o[e] / L : 0.f;
  }
  if (tid == 0) a.counters[b * n_hg + hg] = 0u;
}

}  // namespace g4
