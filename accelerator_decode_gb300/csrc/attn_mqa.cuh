// Decode attention for one KV head shared by all query heads (MQA), one CTA per (split,
// sequence) serving every query head from one load of each K/V tile.
//
// Same computation as attn_unit (attn.cuh): per sequence b at position p, for each query head
// h, q_h = RoPE(RMSNorm(q_raw_h) g_q); owning layers write the new K/V row at (slot, p); keys
// j in [lo, p]; s_hj = scale q_h . K_j; o_h = sum_j softmax_j(s_h) V_j; splits merged by their
// log-sum-exp.  With eight query heads over one KV head ("Porting Gemma 4 E2B to SGLang-JAX",
// Step 1: num_kv_heads = 1), a CTA per (split, head) fetches every tile eight times (from L2)
// and walks the keys of one head serially; here a tile of 32 keys is staged once and
//   scores:  warp w takes the d-slice [w D/8, (w+1) D/8) of all 32 keys (lane = key) against
//            every head's q (shared-memory broadcasts), partial sums reduced across warps;
//   softmax: warp h takes head h (lane = key), online max / sum in registers;
//   P V:     thread t owns output dims [t PT, (t+1) PT) of every head.
// Tile rows are padded by 16 bytes so that the 32 lanes' row reads hit distinct banks.
#pragma once
#include "attn.cuh"

namespace g4 {

constexpr int kMqaThreads = 256;
constexpr int kMqaWarps = kMqaThreads / 32;
constexpr int kMqaMaxHeads = 8;

template <int D, bool KV8>
struct MqaLayout {
  static constexpr int EB = KV8 ? 1 : 2;                 // bytes per cached value
  static constexpr int ROW = D * EB + 16;                // padded tile row, bytes
  static constexpr int TILE_BYTES = kAttnTile * ROW;
};

template <int D, bool KV8>
__host__ __device__ inline size_t mqa_smem_bytes(int nstage) {
  using Ly = MqaLayout<D, KV8>;
  return (size_t)nstage * 2 * Ly::TILE_BYTES                     // K, V tiles
         + (KV8 ? (size_t)nstage * 2 * kAttnTile * 4 : 0)         // their row scales
         + ((size_t)kMqaMaxHeads * D + 2 * D                       // q, new k / v
            + (size_t)kMqaWarps * kMqaMaxHeads * kAttnTile          // score partials
            + kMqaMaxHeads * kAttnTile + 3 * kMqaMaxHeads           // weights, rescale, m, l
            + 64 + 4 + 4) * 4;                                      // merge weights, flag, new scales
}

template <int D, bool KV8>
__global__ void __launch_bounds__(kMqaThreads) attn_mqa_kernel(const AttnArgs a) {
  using Ly = MqaLayout<D, KV8>;
  constexpr int EB = Ly::EB, ROW = Ly::ROW, TB = Ly::TILE_BYTES;
  constexpr int CH = D / kMqaWarps;                              // score d-slice per warp
  constexpr int PT = D >= kMqaThreads ? D / kMqaThreads : 1;     // output dims per thread
  constexpr int PT2 = 1;                                         // float2 accumulators per head
  static_assert(PT <= 2, "head dim up to 512");
  static_assert(D % 64 == 0 && CH % 8 == 0, "head dim must be a multiple of 64");
  extern __shared__ __align__(16) unsigned char msm[];
  unsigned char* Ks = msm;
  unsigned char* Vs = Ks + (size_t)a.nstage * TB;
  float* Kss = reinterpret_cast<float*>(Vs + (size_t)a.nstage * TB);
  float* Vss = Kss + (KV8 ? a.nstage * kAttnTile : 0);
  float* qs = Vss + (KV8 ? a.nstage * kAttnTile : 0);   // [heads][D]
  float* knew = qs + kMqaMaxHeads * D;
  float* vnew = knew + D;
  float* part = vnew + D;                               // [warps][heads][TILE]
  float* ps = part + kMqaWarps * kMqaMaxHeads * kAttnTile;  // [heads][TILE]
  float* resc = ps + kMqaMaxHeads * kAttnTile;
  float* m_sh = resc + kMqaMaxHeads;
  float* l_sh = m_sh + kMqaMaxHeads;
  float* wgt = l_sh + kMqaMaxHeads;                     // [64]
  int* is_last_p = reinterpret_cast<int*>(wgt + 64);
  float* kvs_new = wgt + 68;                            // KV8: scales of the new K and V rows

  const int split = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nq = a.nq;

  int p = __ldcg(a.positions + b);
  const int slot = __ldcg(a.slots + b);
  bool bad = false;
  if (p < 0 || p >= a.t_max) { if (split == 0 && tid == 0) set_err(a.err, G4_DEV_BAD_POSITION); bad = true; }
  if (slot < 0 || slot >= a.max_batch) { if (split == 0 && tid == 0) set_err(a.err, G4_DEV_BAD_SLOT); bad = true; }
  if (bad) p = -1;
  const int lo = (p < 0) ? 0 : (a.window > 0 ? max(0, p - a.window + 1) : 0);
  const int nkeys = p - lo + 1;  // 0 when bad
  const int chunk = nkeys > 0 ? ((nkeys + a.nsplit - 1) / a.nsplit + kAttnTile - 1) / kAttnTile * kAttnTile : 0;
  const int j0 = lo + split * chunk;
  const int j1 = min(p + 1, j0 + chunk);
  const bool has_p = (p >= 0) && (j0 <= p) && (p < j1);
  const int ntiles = j1 > j0 ? (j1 - j0 + kAttnTile - 1) / kAttnTile : 0;
  const unsigned char* kbase = reinterpret_cast<const unsigned char*>(a.kc);
  const unsigned char* vbase = reinterpret_cast<const unsigned char*>(a.vc);
  const int slot0 = slot < 0 ? 0 : slot;
  if (!a.early) {  // the previous kernel wrote cache rows this launch reads
    pdl_wait();
    pdl_trigger();
  }

  // tile loader: keys [t0, t0 + 32) clipped to j1; rows past it (or without a page) are
  // zero-filled, with zero scales
  auto load_tile = [&](int ti) {
    const int t0 = j0 + ti * kAttnTile;
    const int st = ti % a.nstage;
    constexpr int CR = D * EB / 16;  // 16-byte chunks per row
    for (int i = tid; i < kAttnTile * CR; i += kMqaThreads) {
      const int r = i / CR, c = i - r * CR;
      const long row = t0 + r < j1 ? kv_row_index(a, slot0, t0 + r) : -1L;
      const bool ok = row >= 0;
      if (!ok && c == 0 && t0 + r < j1) set_err(a.err, G4_DEV_BAD_POSITION);  // no page
      const size_t off = (size_t)(ok ? row : 0) * D * EB + 16 * c;
      cp_async16(Ks + (size_t)st * TB + r * ROW + 16 * c, kbase + off, ok);
      cp_async16(Vs + (size_t)st * TB + r * ROW + 16 * c, vbase + off, ok);
      if constexpr (KV8) {
        if (c == 0) {
          if (ok) {
            cp_async4(Kss + st * kAttnTile + r, a.ksc + row);
            cp_async4(Vss + st * kAttnTile + r, a.vsc + row);
          } else {
            Kss[st * kAttnTile + r] = 0.f;
            Vss[st * kAttnTile + r] = 0.f;
          }
        }
      }
    }
    asm volatile("cp.async.commit_group;\n" ::: "memory");
  };
  if (ntiles > 0) load_tile(0);
  if (ntiles > 1 && a.nstage > 1) load_tile(1);
  // in a decode step, cache rows, positions, slots and page tables were final before this
  // launch (the new row of an owning layer is patched in from registers): the first tiles go
  // out before waiting for the previous kernel, whose output (q) is read after it
  if (a.early) {
    pdl_wait();
    pdl_trigger();
  }

  // ---- q of every head (warp per head): RMSNorm, gain, RoPE at p; then the new K/V row
  const float* qraw = a.qkv + (size_t)b * a.qkv_stride;
  const bool use_new = a.own && has_p;
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
    for (int h = warp; h < nq; h += kMqaWarps) {
      const float* src = qraw + (size_t)h * D;
      float qv[D / 32];
#pragma unroll
      for (int e = 0; e < D / 32; ++e) qv[e] = __ldcg(src + lane + 32 * e);  // written by another grid
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
      for (int e = 0; e < D / 32; ++e) qs[h * D + lane + 32 * e] = qv[e];
    }
  }
  if (use_new && warp == 0) kv_row<D, KV8>(a, qraw, slot, p, cs, sn, knew, vnew, kvs_new, true);

  // ---- tiles with online softmax.  Heads past nq run on zero queries (their weights are
  // zeroed) so that every loop below has a fixed trip count.
  for (int i = nq * D + tid; i < kMqaMaxHeads * D; i += kMqaThreads) qs[i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // head `warp` (warps < nq)
  float2 acc[kMqaMaxHeads][PT2];
#pragma unroll
  for (int h = 0; h < kMqaMaxHeads; ++h)
#pragma unroll
    for (int e = 0; e < PT2; ++e) acc[h][e] = make_float2(0.f, 0.f);

  for (int ti = 0; ti < ntiles; ++ti) {
    const int t0 = j0 + ti * kAttnTile;
    const int tn = min(kAttnTile, j1 - t0);
    const int st = ti % a.nstage;
    if (a.nstage > 1 && ti + 1 < ntiles) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
    else asm volatile("cp.async.wait_group 0;\n" ::: "memory");
    __syncthreads();
    unsigned char* Kt = Ks + (size_t)st * TB;
    unsigned char* Vt = Vs + (size_t)st * TB;
    if (use_new && p >= t0 && p < t0 + kAttnTile) {
      // the new row (computed above, maybe not yet in the cache when the tile was fetched)
      const int r = p - t0;
      for (int d = tid; d < D; d += kMqaThreads) {
        if constexpr (KV8) {
          reinterpret_cast<int8_t*>(Kt + r * ROW)[d] = (int8_t)knew[d];
          reinterpret_cast<int8_t*>(Vt + r * ROW)[d] = (int8_t)vnew[d];
        } else {
          reinterpret_cast<__nv_bfloat16*>(Kt + r * ROW)[d] = __float2bfloat16_rn(knew[d]);
          reinterpret_cast<__nv_bfloat16*>(Vt + r * ROW)[d] = __float2bfloat16_rn(vnew[d]);
        }
      }
      if (KV8 && tid == 0) {
        Kss[st * kAttnTile + r] = kvs_new[0];
        Vss[st * kAttnTile + r] = kvs_new[1];
      }
      __syncthreads();
    }
    // scores: this warp's d-slice of key `lane` against every head (pairs of dims)
    {
      float2 kr[CH / 2];
      if constexpr (KV8) {
        const unsigned char* kp = Kt + lane * ROW + warp * CH;
        if constexpr (CH >= 16) {
#pragma unroll
          for (int v = 0; v < CH / 16; ++v) {
            const uint4 u = reinterpret_cast<const uint4*>(kp)[v];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              kr[8 * v + 2 * m] = make_float2(i8f(w[m], 0), i8f(w[m], 1));
              kr[8 * v + 2 * m + 1] = make_float2(i8f(w[m], 2), i8f(w[m], 3));
            }
          }
        } else {
          const uint2 u = *reinterpret_cast<const uint2*>(kp);
          kr[0] = make_float2(i8f(u.x, 0), i8f(u.x, 1));
          kr[1] = make_float2(i8f(u.x, 2), i8f(u.x, 3));
          kr[2] = make_float2(i8f(u.y, 0), i8f(u.y, 1));
          kr[3] = make_float2(i8f(u.y, 2), i8f(u.y, 3));
        }
      } else {
        const unsigned char* kp = Kt + lane * ROW + warp * CH * 2;
#pragma unroll
        for (int v = 0; v < CH / 8; ++v) {
          const uint4 u = reinterpret_cast<const uint4*>(kp)[v];
          kr[4 * v + 0] = make_float2(bf16_lo(u.x), bf16_hi(u.x));
          kr[4 * v + 1] = make_float2(bf16_lo(u.y), bf16_hi(u.y));
          kr[4 * v + 2] = make_float2(bf16_lo(u.z), bf16_hi(u.z));
          kr[4 * v + 3] = make_float2(bf16_lo(u.w), bf16_hi(u.w));
        }
      }
#pragma unroll
      for (int h = 0; h < kMqaMaxHeads; ++h) {
        const float4* q4 = reinterpret_cast<const float4*>(qs + h * D + warp * CH);
        float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < CH / 4; ++c) {
          const float4 qv = q4[c];
          d2 = __ffma2_rn(make_float2(qv.x, qv.y), kr[2 * c], d2);
          d2 = __ffma2_rn(make_float2(qv.z, qv.w), kr[2 * c + 1], d2);
        }
        part[(warp * kMqaMaxHeads + h) * kAttnTile + lane] = d2.x + d2.y;
      }
    }
    __syncthreads();
    // softmax statistics: warp h, lane = key; weights of heads past nq and keys past tn are 0
    {
      const int h = warp;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kMqaWarps; ++w) s += part[(w * kMqaMaxHeads + h) * kAttnTile + lane];
      s *= a.scale;
      if constexpr (KV8) s *= Kss[st * kAttnTile + lane];
      const bool live = lane < tn && h < nq;
      if (!live) s = -INFINITY;
      const float mt = warp_max(s);
      const float mn = fmaxf(m_run, mt);
      const float pj = live ? expf(s - mn) : 0.f;
      const float ls = warp_sum(pj);
      const float r = h < nq ? expf(m_run - mn) : 1.f;  // 0 on the first tile
      if constexpr (KV8)  // the value row's scale rides on its weight
        ps[h * kAttnTile + lane] = pj * Vss[st * kAttnTile + lane];
      else
        ps[h * kAttnTile + lane] = pj;
      if (lane == 0) resc[h] = r;
      if (h < nq) {
        m_run = mn;
        l_run = l_run * r + ls;
      }
    }
    __syncthreads();
    // P V: thread owns dims [tid * PT, +PT) of every head; keys four at a time (rows past tn
    // are zero with zero weight)
    if (tid * PT < D) {
#pragma unroll
      for (int h = 0; h < kMqaMaxHeads; ++h) {
        const float r = resc[h];
#pragma unroll
        for (int e = 0; e < PT2; ++e) { acc[h][e].x *= r; acc[h][e].y *= r; }
      }
      const int tn4 = (tn + 3) & ~3;
      for (int jj = 0; jj < tn4; jj += 4) {
        // values of the four keys at this thread's dims
        float vv[4][PT];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if constexpr (KV8) {
            const unsigned char* vp = Vt + (jj + k) * ROW + tid * PT;
            if constexpr (PT == 2) {
              const uint32_t w = *reinterpret_cast<const uint16_t*>(vp);
              vv[k][0] = i8f(w, 0);
              vv[k][1] = i8f(w, 1);
            } else {
              vv[k][0] = i8f(vp[0], 0);
            }
          } else {
            const unsigned char* vp = Vt + (jj + k) * ROW + tid * PT * 2;
            if constexpr (PT == 2) {
              const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
              vv[k][0] = bf16_lo(w);
              vv[k][1] = bf16_hi(w);
            } else {
              vv[k][0] = bf16f(*reinterpret_cast<const __nv_bfloat16*>(vp));
            }
          }
        }
#pragma unroll
        for (int h = 0; h < kMqaMaxHeads; ++h) {
          const float4 pw = *reinterpret_cast<const float4*>(ps + h * kAttnTile + jj);
          if constexpr (PT == 2) {  // (dim 0, dim 1) pairs, one key at a time
            acc[h][0] = __ffma2_rn(make_float2(pw.x, pw.x), make_float2(vv[0][0], vv[0][1]), acc[h][0]);
            acc[h][0] = __ffma2_rn(make_float2(pw.y, pw.y), make_float2(vv[1][0], vv[1][1]), acc[h][0]);
            acc[h][0] = __ffma2_rn(make_float2(pw.z, pw.z), make_float2(vv[2][0], vv[2][1]), acc[h][0]);
            acc[h][0] = __ffma2_rn(make_float2(pw.w, pw.w), make_float2(vv[3][0], vv[3][1]), acc[h][0]);
          } else {  // (even key, odd key) pairs of one dim, added at the end
            acc[h][0] = __ffma2_rn(make_float2(pw.x, pw.y), make_float2(vv[0][0], vv[1][0]), acc[h][0]);
            acc[h][0] = __ffma2_rn(make_float2(pw.z, pw.w), make_float2(vv[2][0], vv[3][0]), acc[h][0]);
          }
        }
      }
    }
    __syncthreads();
    if (a.nstage > 1 && ti + 2 < ntiles) load_tile(ti + 2);
    else if (a.nstage == 1 && ti + 1 < ntiles) load_tile(ti + 1);
  }
  // per-thread output values: PT == 2 keeps (dim 0, dim 1), PT == 1 the two key halves' sum
  float accf[kMqaMaxHeads][PT];
#pragma unroll
  for (int h = 0; h < kMqaMaxHeads; ++h) {
    if constexpr (PT == 2) { accf[h][0] = acc[h][0].x; accf[h][1] = acc[h][0].y; }
    else accf[h][0] = acc[h][0].x + acc[h][0].y;
  }
  if (warp < nq && lane == 0) { m_sh[warp] = m_run; l_sh[warp] = l_run; }
  __syncthreads();

  float* outb = a.out + (size_t)b * a.out_stride;
  if (a.nsplit == 1) {
    if (tid * PT < D) {
#pragma unroll
      for (int h = 0; h < kMqaMaxHeads; ++h) {
        if (h < nq) {
          const float L = l_sh[h];
#pragma unroll
          for (int e = 0; e < PT; ++e) outb[h * D + tid * PT + e] = L > 0.f ? accf[h][e] / L : 0.f;
        }
      }
    }
    return;
  }
  // partial -> scratch
  const size_t base_ml = ((size_t)b * nq) * a.nsplit;
#pragma unroll
  for (int h = 0; h < kMqaMaxHeads; ++h) {
    if (h < nq) {
      const size_t row = base_ml + (size_t)h * a.nsplit + split;
      if (tid == 0) { a.ws_ml[row * 2] = m_sh[h]; a.ws_ml[row * 2 + 1] = l_sh[h]; }
      if (tid * PT < D) {
#pragma unroll
        for (int e = 0; e < PT; ++e) a.ws_o[row * D + tid * PT + e] = accf[h][e];
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *is_last_p = atomicAdd(&a.counters[b], 1u) == (unsigned)a.nsplit - 1;
  __syncthreads();
  if (!*is_last_p) return;
  __threadfence();
  // merge: w_s = exp(m_s - M) per split (empty splits carry l = 0 and o = 0), then
  // o = sum_s w_s o_s / sum_s w_s l_s; warp h computes head h's weights
  float* wg = part;  // [heads][64] reuses the score partials (free after the loop)
  for (int h = warp; h < nq; h += kMqaWarps) {
    const size_t row0 = base_ml + (size_t)h * a.nsplit;
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
      if (s < a.nsplit) wg[h * 64 + s] = w;
      L += w * lv[u];
    }
    L = warp_sum(L);
    if (lane == 0) l_sh[h] = L;
  }
  __syncthreads();
  if (tid * PT < D) {
    // every head's partial of a split is loaded before any is used: one round trip per split
    float o[kMqaMaxHeads][PT];
#pragma unroll
    for (int h = 0; h < kMqaMaxHeads; ++h)
#pragma unroll
      for (int e = 0; e < PT; ++e) o[h][e] = 0.f;
    for (int s = 0; s < a.nsplit; ++s) {
      float v[kMqaMaxHeads][PT];
#pragma unroll
      for (int h = 0; h < kMqaMaxHeads; ++h)
#pragma unroll
        for (int e = 0; e < PT; ++e)
          v[h][e] = h < nq ? ldcg(a.ws_o + (base_ml + (size_t)h * a.nsplit + s) * D + tid * PT + e) : 0.f;
#pragma unroll
      for (int h = 0; h < kMqaMaxHeads; ++h) {
        const float w = h < nq ? wg[h * 64 + s] : 0.f;
#pragma unroll
        for (int e = 0; e < PT; ++e) o[h][e] += w * v[h][e];
      }
    }
#pragma unroll
    for (int h = 0; h < kMqaMaxHeads; ++h) {
      if (h < nq) {
        const float L = l_sh[h];
#pragma unroll
        for (int e = 0; e < PT; ++e) outb[h * D + tid * PT + e] = L > 0.f ? o[h][e] / L : 0.f;
      }
    }
  }
  if (tid == 0) a.counters[b] = 0u;
}

}  // namespace g4
