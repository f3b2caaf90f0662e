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
// The visible keys are cut into nsplit chunks (one CTA each), staged through shared memory
// in tiles of 32 keys (2-stage cp.async pipeline) and reduced with an online softmax; the
// last CTA of a (sequence, head group) merges the chunks with their log-sum-exp weights.
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
  int nstage;              // 1 or 2 tile buffers
  float* ws_ml;            // [nb][nq][nsplit][2]
  float* ws_o;             // [nb][nq][nsplit][D]
  unsigned* counters;      // [nb][nq / HPC]
  int* err;
};

template <int D, int HPC>
__host__ __device__ inline size_t attn_smem_bytes(int nstage) {
  return (size_t)nstage * 2 * kAttnTile * D * 2                      // K, V tiles (bf16)
         + ((size_t)HPC * D + 2 * D + HPC * kAttnTile + 4 * HPC) * 4   // q, new k/v, scores, stats
         + (64 + 4) * 4;                                             // merge weights, last flag
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// New K/V row of an owning layer at position p, on one warp: k = RoPE(RMSNorm(k) g_k), v,
// both rounded to bf16.  Stores the row in the cache when `store`; copies the rounded values
// to knew / vnew (shared, [D]) when they are given.  cs / sn: this lane's RoPE factors at p.
template <int D>
__device__ __forceinline__ void kv_row(const AttnArgs& a, const float* qraw, int slot, int p, const float (&cs)[D / 64],
                                       const float (&sn)[D / 64], float* knew, float* vnew, bool store) {
  const int lane = threadIdx.x & 31;
  const float* kr = qraw + (size_t)a.nq * D;
  const float* vr = kr + D;
  float kv_[D / 32], vv_[D / 32], gk[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) {
    kv_[e] = __ldcg(kr + lane + 32 * e);
    vv_[e] = __ldcg(vr + lane + 32 * e);
    gk[e] = bf16f(a.g_k[lane + 32 * e]);
  }
  float ss = 0.f;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) ss += kv_[e] * kv_[e];
  ss = warp_sum(ss);
  const float den = rms_denom(ss, D, a.eps);
#pragma unroll
  for (int e = 0; e < D / 32; ++e) kv_[e] = (kv_[e] / den) * gk[e];
  __nv_bfloat16* kdst = a.kc + ((size_t)slot * a.t_max + p) * D;
  __nv_bfloat16* vdst = a.vc + ((size_t)slot * a.t_max + p) * D;
#pragma unroll
  for (int e = 0; e < D / 64; ++e) {
    const int i = lane + 32 * e;
    const float ka = kv_[e], kb = kv_[e + D / 64];
    const __nv_bfloat16 k1 = __float2bfloat16_rn(ka * cs[e] - kb * sn[e]);
    const __nv_bfloat16 k2 = __float2bfloat16_rn(kb * cs[e] + ka * sn[e]);
    if (knew) { knew[i] = bf16f(k1); knew[i + D / 2] = bf16f(k2); }
    if (store) { kdst[i] = k1; kdst[i + D / 2] = k2; }
  }
#pragma unroll
  for (int e = 0; e < D / 32; ++e) {
    const __nv_bfloat16 v1 = __float2bfloat16_rn(vv_[e]);
    if (vnew) vnew[lane + 32 * e] = bf16f(v1);
    if (store) vdst[lane + 32 * e] = v1;
  }
}

// One (split, head group, sequence) unit on kAttnThreads threads; `asmem` holds
// attn_smem_bytes<D, HPC>(a.nstage) bytes.  Called by attn_kernel and by the persistent step.
template <int D, int HPC>
// Threads [tid_base, tid_base + 128) run the unit and synchronise on named barrier bar_id.
__device__ __forceinline__ void attn_unit(const AttnArgs& a, int split, int hg, int b, unsigned char* asmem,
                                          int tid_base, int bar_id) {
  constexpr int PL = D / 32;                                    // q/k elements per lane (scores)
  constexpr int PT = D >= kAttnThreads ? D / kAttnThreads : 1;  // output elements per thread
  static_assert(PL >= 2 && PL % 2 == 0, "head dim must be a multiple of 64");
  constexpr int TD = kAttnTile * D;
  __nv_bfloat16* Ks = reinterpret_cast<__nv_bfloat16*>(asmem);  // [nstage][TILE][D]
  __nv_bfloat16* Vs = Ks + (size_t)a.nstage * TD;                // [nstage][TILE][D]
  float* qs = reinterpret_cast<float*>(Vs + (size_t)a.nstage * TD);  // [HPC][D]
  float* knew = qs + HPC * D;
  float* vnew = knew + D;
  float* sc = vnew + D;          // [HPC][TILE]
  float* resc = sc + HPC * kAttnTile;
  float* m_sh = resc + HPC;
  float* l_sh = m_sh + HPC;
  float* wgt = l_sh + 2 * HPC;                           // [64]
  int* is_last_p = reinterpret_cast<int*>(wgt + 64);

  const int tid = threadIdx.x - tid_base, warp = tid >> 5, lane = tid & 31;
  const int h0 = hg * HPC;
  const int n_hg = a.nq / HPC;

  int p = __ldcg(a.positions + b);
  const int slot = __ldcg(a.slots + b);
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
  const int ntiles = j1 > j0 ? (j1 - j0 + kAttnTile - 1) / kAttnTile : 0;
  const __nv_bfloat16* kbase = a.kc + (size_t)(slot < 0 ? 0 : slot) * a.t_max * D;
  const __nv_bfloat16* vbase = a.vc + (size_t)(slot < 0 ? 0 : slot) * a.t_max * D;

  // tile loader: keys [t0, t0 + 32) clipped to j1; rows past it are zero-filled
  auto load_tile = [&](int ti) {
    const int t0 = j0 + ti * kAttnTile;
    const int st = ti % a.nstage;
    constexpr int C8 = D / 8;  // 16-byte chunks per row
    for (int i = tid; i < kAttnTile * C8; i += kAttnThreads) {
      const int r = i / C8, c = i - r * C8;
      const bool ok = t0 + r < j1;
      const size_t off = (size_t)(ok ? t0 + r : 0) * D + 8 * c;
      cp_async16(Ks + (size_t)st * TD + r * D + 8 * c, kbase + off, ok);
      cp_async16(Vs + (size_t)st * TD + r * D + 8 * c, vbase + off, ok);
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
  if (ntiles > 0) load_tile(0);
  if (ntiles > 1 && a.nstage > 1) load_tile(1);

  // ---- q: per-head RMSNorm then RoPE at position p, in registers.  Every global value is
  // loaded before the first shared-memory store: a load issued after a store through another
  // pointer may not be moved above it, which would serialise one L2 round trip per element.
  // RoPE pairs element i with i + D/2; for i = lane + 32 e (e < D/64) the partner is
  // lane + 32 (e + D/64), so both halves of a pair sit in the same lane.
  const float* qraw = a.qkv + (size_t)b * a.qkv_stride;
  const bool use_new = a.own && has_p;
  constexpr int kKvWarp = kAttnThreads / 32 - 1;  // computes the new K/V row beside the q warps
  float cs[D / 64], sn[D / 64];
  if (ntiles > 0 || use_new) {
    const size_t rp = (size_t)(p < 0 ? 0 : p) * (D / 2);
#pragma unroll
    for (int e = 0; e < D / 64; ++e) {
      cs[e] = __ldg(a.rope_cos + rp + lane + 32 * e);
      sn[e] = __ldg(a.rope_sin + rp + lane + 32 * e);
    }
  }
  if (ntiles > 0) {
    float gq[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) gq[e] = bf16f(a.g_q[lane + 32 * e]);
    for (int hh = warp; hh < HPC; hh += kAttnThreads / 32) {
      const float* src = qraw + (size_t)(h0 + hh) * D;
      float qv[D / 32];
#pragma unroll
      for (int e = 0; e < D / 32; ++e) qv[e] = __ldcg(src + lane + 32 * e);  // written by another grid/CTA
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) ss += qv[e] * qv[e];
      ss = warp_sum(ss);
      const float den = rms_denom(ss, D, a.eps);
#pragma unroll
      for (int e = 0; e < D / 32; ++e) qv[e] = (qv[e] / den) * gq[e];
#pragma unroll
      for (int e = 0; e < D / 64; ++e) {
        const float qa = qv[e], qb = qv[e + D / 64];
        qv[e] = qa * cs[e] - qb * sn[e];
        qv[e + D / 64] = qb * cs[e] + qa * sn[e];
      }
#pragma unroll
      for (int e = 0; e < D / 32; ++e) qs[hh * D + lane + 32 * e] = qv[e];
    }
  }
  // ---- new K/V row of an owning layer (position p), computed by every CTA holding key p
  if (use_new && warp == kKvWarp) kv_row<D>(a, qraw, slot, p, cs, sn, knew, vnew, hg == 0);

  // ---- tiles with online softmax
  float m_run[HPC], l_run[HPC];
  float acc[HPC][PT];
#pragma unroll
  for (int h = 0; h < HPC; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < PT; ++e) acc[h][e] = 0.f;
  }
  for (int ti = 0; ti < ntiles; ++ti) {
    const int t0 = j0 + ti * kAttnTile;
    const int tn = min(kAttnTile, j1 - t0);
    const int st = ti % a.nstage;
    if (a.nstage > 1 && ti + 1 < ntiles) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    else asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    named_sync(bar_id, kAttnThreads);
    const __nv_bfloat16* Kt = Ks + (size_t)st * TD;
    const __nv_bfloat16* Vt = Vs + (size_t)st * TD;
    // scores: warp per key, lanes over D.  A warp's keys (jj = warp + 4 q) are dotted first and
    // reduced together, so the shuffle chains overlap; zero-filled rows past tn are skipped.
    constexpr int KPW = kAttnTile / (kAttnThreads / 32);
    float qreg[PL];
    if constexpr (HPC == 1) {
#pragma unroll
      for (int e = 0; e < PL; ++e) qreg[e] = qs[lane * PL + e];
    }
    float dq[HPC][KPW];
#pragma unroll
    for (int q = 0; q < KPW; ++q) {
      const int jj = warp + q * (kAttnThreads / 32);
      const int j = t0 + jj;
#pragma unroll
      for (int h = 0; h < HPC; ++h) dq[h][q] = 0.f;
      if (jj >= tn) continue;
      float kv[PL];
      if (use_new && j == p) {
#pragma unroll
        for (int e = 0; e < PL; ++e) kv[e] = knew[lane * PL + e];
      } else if constexpr (PL % 8 == 0) {
#pragma unroll
        for (int c = 0; c < PL / 8; ++c) {
          const uint4 u = reinterpret_cast<const uint4*>(Kt + jj * D + lane * PL)[c];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int m = 0; m < 4; ++m) { kv[c * 8 + 2 * m] = bf16_lo(w[m]); kv[c * 8 + 2 * m + 1] = bf16_hi(w[m]); }
        }
      } else {
#pragma unroll
        for (int c = 0; c < PL / 2; ++c) {
          const uint32_t w = reinterpret_cast<const uint32_t*>(Kt + jj * D + lane * PL)[c];
          kv[2 * c] = bf16_lo(w);
          kv[2 * c + 1] = bf16_hi(w);
        }
      }
#pragma unroll
      for (int h = 0; h < HPC; ++h) {
        float d = 0.f;
        if constexpr (HPC == 1) {
#pragma unroll
          for (int e = 0; e < PL; ++e) d += qreg[e] * kv[e];
        } else {
#pragma unroll
          for (int e = 0; e < PL; ++e) d += qs[h * D + lane * PL + e] * kv[e];
        }
        dq[h][q] = d;
      }
    }
#pragma unroll
    for (int q = 0; q < KPW; ++q)
#pragma unroll
      for (int h = 0; h < HPC; ++h) dq[h][q] = warp_sum(dq[h][q]);
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < KPW; ++q) {
        const int jj = warp + q * (kAttnThreads / 32);
#pragma unroll
        for (int h = 0; h < HPC; ++h) sc[h * kAttnTile + jj] = (jj < tn) ? dq[h][q] * a.scale : -INFINITY;
      }
    }
    named_sync(bar_id, kAttnThreads);
    // softmax statistics per head (warp per head)
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
      if ((h % (kAttnThreads / 32)) != warp) continue;
      const float s = sc[h * kAttnTile + lane];
      const float mt = warp_max(s);
      const float mn = fmaxf(m_run[h], mt);
      const float pj = (lane < tn) ? expf(s - mn) : 0.f;
      const float ls = warp_sum(pj);
      const float r = expf(m_run[h] - mn);  // 0 on the first tile
      sc[h * kAttnTile + lane] = pj;
      if (lane == 0) resc[h] = r;
      m_run[h] = mn;
      l_run[h] = l_run[h] * r + ls;
    }
    named_sync(bar_id, kAttnThreads);
    // P V: thread owns PT contiguous elements of each head's output
    if (tid * PT < D) {
#pragma unroll
      for (int h = 0; h < HPC; ++h) {
        const float r = resc[h];
#pragma unroll
        for (int e = 0; e < PT; ++e) acc[h][e] *= r;
      }
#pragma unroll 4
      for (int jj = 0; jj < tn; ++jj) {
        const int j = t0 + jj;
        float vv[PT];
        if (use_new && j == p) {
#pragma unroll
          for (int e = 0; e < PT; ++e) vv[e] = vnew[tid * PT + e];
        } else {
          const __nv_bfloat16* vp = Vt + jj * D + tid * PT;
          if constexpr (PT == 1) {
            vv[0] = bf16f(vp[0]);
          } else if constexpr (PT == 2) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
            vv[0] = bf16_lo(w);
            vv[1] = bf16_hi(w);
          } else {
            const uint2 w = *reinterpret_cast<const uint2*>(vp);
            vv[0] = bf16_lo(w.x); vv[1] = bf16_hi(w.x); vv[2] = bf16_lo(w.y); vv[3] = bf16_hi(w.y);
          }
        }
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
          const float pj = sc[h * kAttnTile + jj];
#pragma unroll
          for (int e = 0; e < PT; ++e) acc[h][e] += pj * vv[e];
        }
      }
    }
    named_sync(bar_id, kAttnThreads);
    if (a.nstage > 1 && ti + 2 < ntiles) load_tile(ti + 2);
    else if (a.nstage == 1 && ti + 1 < ntiles) load_tile(ti + 1);
  }
#pragma unroll
  for (int h = 0; h < HPC; ++h)
    if ((h % (kAttnThreads / 32)) == warp && lane == 0) { m_sh[h] = m_run[h]; l_sh[h] = l_run[h]; }
  named_sync(bar_id, kAttnThreads);

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
  named_sync(bar_id, kAttnThreads);
  if (tid == 0) *is_last_p = atomicAdd(&a.counters[b * n_hg + hg], 1u) == (unsigned)a.nsplit - 1;
  named_sync(bar_id, kAttnThreads);
  if (!*is_last_p) return;
  __threadfence();
  // merge: w_s = exp(m_s - M) per split (empty splits carry l = 0 and o = 0), then
  // o = sum_s w_s o_s / sum_s w_s l_s
  for (int h = 0; h < HPC; ++h) {
    const size_t row0 = base_ml + (size_t)(h0 + h) * a.nsplit;
    if (warp == 0) {
      float mv[2], lv[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int s = lane + 32 * u;
        mv[u] = -INFINITY;
        lv[u] = 0.f;
        if (s < a.nsplit) { mv[u] = ldcg(a.ws_ml + (row0 + s) * 2); lv[u] = ldcg(a.ws_ml + (row0 + s) * 2 + 1); }
      }
      float M = -INFINITY;
#pragma unroll
      for (int u = 0; u < 2; ++u) if (lv[u] > 0.f) M = fmaxf(M, mv[u]);
      M = warp_max(M);
      float L = 0.f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int s = lane + 32 * u;
        const float w = (lv[u] > 0.f) ? expf(mv[u] - M) : 0.f;
        if (s < a.nsplit) wgt[s] = w;
        L += w * lv[u];
      }
      L = warp_sum(L);
      if (lane == 0) l_sh[h] = L;
    }
    named_sync(bar_id, kAttnThreads);
    const float L = l_sh[h];
    if (tid * PT < D) {
      float o[PT];
#pragma unroll
      for (int e = 0; e < PT; ++e) o[e] = 0.f;
#pragma unroll 16
      for (int s = 0; s < a.nsplit; ++s) {
        const float w = wgt[s];
#pragma unroll
        for (int e = 0; e < PT; ++e) o[e] += w * ldcg(a.ws_o + (row0 + s) * D + tid * PT + e);
      }
#pragma unroll
      for (int e = 0; e < PT; ++e) outb[(h0 + h) * D + tid * PT + e] = L > 0.f ? o[e] / L : 0.f;
    }
    named_sync(bar_id, kAttnThreads);
  }
  if (tid == 0) a.counters[b * n_hg + hg] = 0u;
}

template <int D, int HPC>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) unsigned char asmem_k[];
  pdl_wait();
  pdl_trigger();
  attn_unit<D, HPC>(a, blockIdx.x, blockIdx.y, blockIdx.z, asmem_k, 0, 1);
}

// K/V rows of an owning layer for every row of a step before its attention runs (prefill
// blocks: rows of one sequence at consecutive positions read each other's keys, so no row
// may append its own key inside the attention launch).  One warp per row.
template <int D>
__global__ void __launch_bounds__(32) kv_write_kernel(const AttnArgs a) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, lane = threadIdx.x;
  const int p = __ldcg(a.positions + b), slot = __ldcg(a.slots + b);
  if (p < 0 || p >= a.t_max || slot < 0 || slot >= a.max_batch) return;  // attention flags it
  float cs[D / 64], sn[D / 64];
#pragma unroll
  for (int e = 0; e < D / 64; ++e) {
    cs[e] = __ldg(a.rope_cos + (size_t)p * (D / 2) + lane + 32 * e);
    sn[e] = __ldg(a.rope_sin + (size_t)p * (D / 2) + lane + 32 * e);
  }
  kv_row<D>(a, a.qkv + (size_t)b * a.qkv_stride, slot, p, cs, sn, nullptr, nullptr, true);
}

}  // namespace g4
