// Decode attention with one KV head (MQA), split over keys (flash-decode).
//
// Per sequence b at position p, for the query heads of one head group:
//   q_h = RoPE(RMSNorm(q_raw_h) * g_q)                      (every layer)
//   owning layers: k = RoPE(RMSNorm(k_raw) * g_k), v = v_raw written in place at cache row
//   (slot, p) -- a sharing layer applies RoPE to its queries only and reads its source
//   layer's cache ("Porting Gemma 4 E2B to SGLang-JAX", Step 4; "One TPU chip, eight
//   agents", The engine: kv_share_map, static cache written in place).
// Cache rows are bf16, or int8 codes with one fp32 scale per row ("One TPU chip, eight
// agents", Measured: the raw JAX decode kernel, int8 KV cache): s = max|r| / 127,
// c = round-half-even(r / s) clipped to +-127, stored value c * s.  With int8 rows the row
// scale is applied once per key (to the score, and to the softmax weight of the value row).
// Row addresses are static (slot * max_context + position) or paged: page_table[slot][p /
// page_size] names the pool page that holds positions [p - p % page_size, +page_size)
// ("Six serving engines on one Cloud TPU v5e chip", Step 3, page size 128).
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
  int early;               // request the first K/V tiles before the dependency wait (no kernel
                           // right before this one writes cache rows: not behind kv_write_kernel)
  void* kc;                // cache of the source layer: rows of D bf16 or D int8 (KV8)
  void* vc;
  float* ksc;              // KV8: fp32 scale per row
  float* vsc;
  const int* page_table;   // paged: [max_batch][max_pages] pool page per page of positions; NULL: static
  int page_shift;          // log2(page size)
  int max_pages;
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

template <int D, int HPC, bool KV8 = false>
__host__ __device__ inline size_t attn_smem_bytes(int nstage) {
  return (size_t)nstage * 2 * kAttnTile * D * (KV8 ? 1 : 2)          // K, V tiles
         + (KV8 ? (size_t)nstage * 2 * kAttnTile * 4 : 0)            // their row scales
         + ((size_t)HPC * D + 2 * D + HPC * kAttnTile + 4 * HPC) * 4   // q, new k/v, scores, stats
         + (64 + 4 + 4) * 4;                                         // merge weights, last flag, new scales
}

// Cache row of (slot, position j): static, or through the slot's page table; -1 when the
// position has no page.
__device__ __forceinline__ long kv_row_index(const AttnArgs& a, int slot, int j) {
  if (!a.page_table) return (long)slot * a.t_max + j;
  const int pg = __ldg(a.page_table + (size_t)slot * a.max_pages + (j >> a.page_shift));
  return pg < 0 ? -1L : ((long)pg << a.page_shift) + (j & ((1 << a.page_shift) - 1));
}

// Byte i of w as a signed int8 code, exactly, as fp32 (offset binary in a float's mantissa).
__device__ __forceinline__ float i8f(uint32_t w, int i) {
  return __uint_as_float(__byte_perm(w ^ 0x80808080u, 0x4B000000u, 0x7540u | i)) - 8388736.f;
}

// int8 code of a row of D values spread over a warp (element lane + 32 e in v[e]):
// s = max|v| / 127, c = rint(v / s) clipped to +-127 (0 for an all-zero row).
template <int D>
__device__ __forceinline__ float kv_quant_row(float (&v)[D / 32], int8_t (&c)[D / 32]) {
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) m = fmaxf(m, fabsf(v[e]));
  m = warp_max(m);
  const float s = m / 127.f;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) c[e] = s > 0.f ? (int8_t)fminf(fmaxf(rintf(v[e] / s), -127.f), 127.f) : (int8_t)0;
  return s;
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// New K/V row of an owning layer at position p, on one warp: k = RoPE(RMSNorm(k) g_k), v,
// rounded to bf16 or coded to int8.  Stores the row in the cache when `store`; copies the
// stored values to knew / vnew (shared, [D]) when they are given -- for int8 rows the codes,
// with the two row scales in kvs_new[0..1].  cs / sn: this lane's RoPE factors at p.
template <int D, bool KV8>
__device__ __forceinline__ void kv_row(const AttnArgs& a, const float* qraw, int slot, int p, const float (&cs)[D / 64],
                                       const float (&sn)[D / 64], float* knew, float* vnew, float* kvs_new,
                                       bool store) {
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
  // RoPE pairs element i with i + D/2: for i = lane + 32 e (e < D/64) the partner is in
  // kv_[e + D/64] of the same lane
#pragma unroll
  for (int e = 0; e < D / 64; ++e) {
    const float ka = kv_[e], kb = kv_[e + D / 64];
    kv_[e] = ka * cs[e] - kb * sn[e];
    kv_[e + D / 64] = kb * cs[e] + ka * sn[e];
  }
  const long row = kv_row_index(a, slot, p);
  if (row < 0) {
    if (store && lane == 0) set_err(a.err, G4_DEV_BAD_POSITION);
    store = false;
  }
  if constexpr (KV8) {
    int8_t kc8[D / 32], vc8[D / 32];
    const float sk = kv_quant_row<D>(kv_, kc8);
    const float sv = kv_quant_row<D>(vv_, vc8);
    int8_t* kdst = reinterpret_cast<int8_t*>(a.kc) + (size_t)(row < 0 ? 0 : row) * D;
    int8_t* vdst = reinterpret_cast<int8_t*>(a.vc) + (size_t)(row < 0 ? 0 : row) * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      if (knew) { knew[lane + 32 * e] = (float)kc8[e]; vnew[lane + 32 * e] = (float)vc8[e]; }
      if (store) { kdst[lane + 32 * e] = kc8[e]; vdst[lane + 32 * e] = vc8[e]; }
    }
    if (lane == 0) {
      if (kvs_new) { kvs_new[0] = sk; kvs_new[1] = sv; }
      if (store) { a.ksc[row] = sk; a.vsc[row] = sv; }
    }
  } else {
    __nv_bfloat16* kdst = reinterpret_cast<__nv_bfloat16*>(a.kc) + (size_t)(row < 0 ? 0 : row) * D;
    __nv_bfloat16* vdst = reinterpret_cast<__nv_bfloat16*>(a.vc) + (size_t)(row < 0 ? 0 : row) * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
      const __nv_bfloat16 k1 = __float2bfloat16_rn(kv_[e]);
      const __nv_bfloat16 v1 = __float2bfloat16_rn(vv_[e]);
      if (knew) { knew[lane + 32 * e] = bf16f(k1); vnew[lane + 32 * e] = bf16f(v1); }
      if (store) { kdst[lane + 32 * e] = k1; vdst[lane + 32 * e] = v1; }
    }
  }
}

// One (split, head group, sequence) unit on kAttnThreads threads; `asmem` holds
// attn_smem_bytes<D, HPC>(a.nstage) bytes.  Called by attn_kernel and by the persistent step.
template <int D, int HPC, bool KV8 = false>
// Threads [tid_base, tid_base + 128) run the unit and synchronise on named barrier bar_id.
// dep_wait: the unit is a kernel of its own behind a programmatic dependency; it requests its
// first K/V tiles, then waits for the previous kernel (see below).
__device__ __forceinline__ void attn_unit(const AttnArgs& a, int split, int hg, int b, unsigned char* asmem,
                                          int tid_base, int bar_id, bool dep_wait = false) {
  constexpr int PL = D / 32;                                    // q/k elements per lane (scores)
  constexpr int PT = D >= kAttnThreads ? D / kAttnThreads : 1;  // output elements per thread
  static_assert(PL >= 2 && PL % 2 == 0, "head dim must be a multiple of 64");
  constexpr int TD = kAttnTile * D;
  constexpr int EB = KV8 ? 1 : 2;                               // bytes per cached value
  unsigned char* Ks = asmem;                                    // [nstage][TILE][D] values
  unsigned char* Vs = Ks + (size_t)a.nstage * TD * EB;
  float* Kss = reinterpret_cast<float*>(Vs + (size_t)a.nstage * TD * EB);  // KV8: [nstage][TILE] row scales
  float* Vss = Kss + (KV8 ? a.nstage * kAttnTile : 0);
  float* qs = Vss + (KV8 ? a.nstage * kAttnTile : 0);          // [HPC][D]
  float* knew = qs + HPC * D;
  float* vnew = knew + D;
  float* sc = vnew + D;          // [HPC][TILE]
  float* resc = sc + HPC * kAttnTile;
  float* m_sh = resc + HPC;
  float* l_sh = m_sh + HPC;
  float* wgt = l_sh + 2 * HPC;                           // [64]
  int* is_last_p = reinterpret_cast<int*>(wgt + 64);
  float* kvs_new = wgt + 68;                             // KV8: scales of the new K and V rows

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
  const unsigned char* kbase = reinterpret_cast<const unsigned char*>(a.kc);
  const unsigned char* vbase = reinterpret_cast<const unsigned char*>(a.vc);
  const int slot0 = slot < 0 ? 0 : slot;
  if (dep_wait && !a.early) {  // the previous kernel wrote cache rows this unit reads
    pdl_wait();
    pdl_trigger();
  }

  // tile loader: keys [t0, t0 + 32) clipped to j1; rows past it (or without a page) are
  // zero-filled, with zero scales
  auto load_tile = [&](int ti) {
    const int t0 = j0 + ti * kAttnTile;
    const int st = ti % a.nstage;
    constexpr int CR = D * EB / 16;  // 16-byte chunks per row
    for (int i = tid; i < kAttnTile * CR; i += kAttnThreads) {
      const int r = i / CR, c = i - r * CR;
      const long row = t0 + r < j1 ? kv_row_index(a, slot0, t0 + r) : -1L;
      const bool ok = row >= 0;
      if (!ok && c == 0 && t0 + r < j1) set_err(a.err, G4_DEV_BAD_POSITION);  // no page
      const size_t off = (size_t)(ok ? row : 0) * D * EB + 16 * c;
      cp_async16(Ks + ((size_t)st * TD + r * D) * EB + 16 * c, kbase + off, ok);
      cp_async16(Vs + ((size_t)st * TD + r * D) * EB + 16 * c, vbase + off, ok);
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
  // In a decode step the cache rows a unit reads were final before this kernel launched
  // (earlier steps, or the source layer's launch earlier in this step), except the new row of
  // an owning layer, which this kernel writes and substitutes from registers (use_new);
  // positions, slots and page tables are the step's inputs.  So there the first tiles are
  // requested before waiting for the previous kernel; q (its output) and every write come
  // after.
  if (dep_wait && a.early) {
    pdl_wait();
    pdl_trigger();
  }

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
  if (use_new && warp == kKvWarp) kv_row<D, KV8>(a, qraw, slot, p, cs, sn, knew, vnew, kvs_new, hg == 0);

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
    const unsigned char* Kt = Ks + (size_t)st * TD * EB;
    const unsigned char* Vt = Vs + (size_t)st * TD * EB;
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
      } else if constexpr (KV8) {
        const unsigned char* kp = Kt + jj * D + lane * PL;
        if constexpr (PL % 4 == 0) {
#pragma unroll
          for (int c = 0; c < PL / 4; ++c) {
            const uint32_t w = reinterpret_cast<const uint32_t*>(kp)[c];
#pragma unroll
            for (int m = 0; m < 4; ++m) kv[4 * c + m] = i8f(w, m);
          }
        } else {
          const uint32_t w = *reinterpret_cast<const uint16_t*>(kp);
#pragma unroll
          for (int m = 0; m < PL; ++m) kv[m] = i8f(w, m);
        }
      } else if constexpr (PL % 8 == 0) {
#pragma unroll
        for (int c = 0; c < PL / 8; ++c) {
          const uint4 u = reinterpret_cast<const uint4*>(Kt + (jj * D + lane * PL) * 2)[c];
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int m = 0; m < 4; ++m) { kv[c * 8 + 2 * m] = bf16_lo(w[m]); kv[c * 8 + 2 * m + 1] = bf16_hi(w[m]); }
        }
      } else {
#pragma unroll
        for (int c = 0; c < PL / 2; ++c) {
          const uint32_t w = reinterpret_cast<const uint32_t*>(Kt + (jj * D + lane * PL) * 2)[c];
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
        for (int h = 0; h < HPC; ++h) {
          float s_ = dq[h][q] * a.scale;
          if constexpr (KV8) s_ *= (use_new && t0 + jj == p) ? kvs_new[0] : Kss[st * kAttnTile + jj];
          sc[h * kAttnTile + jj] = (jj < tn) ? s_ : -INFINITY;
        }
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
      if constexpr (KV8)  // the value row's scale rides on its weight
        sc[h * kAttnTile + lane] = pj * ((use_new && t0 + lane == p) ? kvs_new[1] : Vss[st * kAttnTile + lane]);
      else
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
        } else if constexpr (KV8) {
          const unsigned char* vp = Vt + jj * D + tid * PT;
          if constexpr (PT == 4) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(vp);
#pragma unroll
            for (int e = 0; e < 4; ++e) vv[e] = i8f(w, e);
          } else if constexpr (PT == 2) {
            const uint32_t w = *reinterpret_cast<const uint16_t*>(vp);
            vv[0] = i8f(w, 0);
            vv[1] = i8f(w, 1);
          } else {
            vv[0] = i8f(vp[0], 0);
          }
        } else {
          const __nv_bfloat16* vp = reinterpret_cast<const __nv_bfloat16*>(Vt) + jj * D + tid * PT;
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

template <int D, int HPC, bool KV8>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) unsigned char asmem_k[];
  attn_unit<D, HPC, KV8>(a, blockIdx.x, blockIdx.y, blockIdx.z, asmem_k, 0, 1, true);
}

// K/V rows of an owning layer for every row of a step before its attention runs (prefill
// blocks: rows of one sequence at consecutive positions read each other's keys, so no row
// may append its own key inside the attention launch).  One warp per row.
template <int D, bool KV8>
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
  kv_row<D, KV8>(a, a.qkv + (size_t)b * a.qkv_stride, slot, p, cs, sn, nullptr, nullptr, nullptr, true);
}

}  // namespace g4
