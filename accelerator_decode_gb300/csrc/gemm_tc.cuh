// Weight-only projections for batches >= 5 on the 5th-generation tensor cores (tcgen05).
//
// D[n, b] = sum_k W[n, k] x[b, k] with the weight rows as the MMA's M (128 per CTA) and the
// padded batch as N ("swap AB").  Per 64-wide k-block:
//   * one thread issues 1-D bulk TMA copies (cp.async.bulk) of the 128 x 64 weight block
//     (int4 GEMV tiles + their bf16 group scales, or bf16 tiles) and of the two activation
//     tiles (x_hi = bf16(x), x_lo = bf16(x - x_hi), pre-swizzled in global memory by the
//     prep kernel) into a 4-stage shared-memory ring, completing on an mbarrier;
//   * 4 dequant warps (one thread per weight row) turn the block into bf16(q * s) -- the same
//     dequantisation as the GEMV ("One TPU chip, eight agents", Two optimizations that
//     didn't work) -- and store it in the 128-byte-swizzled K-major UMMA layout;
//   * one thread issues tcgen05.mma kind::f16 (bf16 x bf16 -> fp32 in TMEM) for both
//     activation parts, and tcgen05.commit releases the stage.
// The epilogue reads the fp32 accumulator with tcgen05.ld.  A K split over CTAs is summed by
// the last CTA of an M tile in split order (deterministic).  Every mbarrier wait is bounded:
// on expiry the CTA sets the device error word, waits (bounded) for its copies in flight,
// frees its TMEM and returns.
#pragma once
#include "common.cuh"
#include "gemv.cuh"

namespace g4 {

constexpr int kTcStages = 4;      // ring stages with a K split (the merge reuses them); 2 without
constexpr int kTcThreads = 192;        // warps 0-3 dequant/epilogue, 4 TMA + TMEM alloc, 5 MMA
constexpr int kTcM = 128;
constexpr int kTcKB = 64;              // k per block
constexpr uint32_t kSpinLimit = 1u << 20;

struct GemmArgs {
  const uint4* qw;       // GEMV tile layout (see gemv.cuh)
  const uint4* sc;       // W4A16 scales (GEMV layout) or nullptr
  int fmt;               // FMT_W4A16 / FMT_BF16
  int tiles, S, n_valid;
  int n_kb;              // k-blocks of 64 over the padded K
  int ksplit, kb_per_split;
  const uint8_t* xt;     // activation tiles [n_kb][2][bpad * 128 bytes]
  int bpad, nb;
  int epi;
  float* y;
  int y_stride;
  const float* ple;
  int ple_stride;
  float* logits;
  int logits_stride;
  float* am_val;         // [nb][gridDim.x]
  int* am_idx;
  float* part;           // [ksplit][n_mtiles * 128 rows][64 columns]
  int stages;            // ring stages: kTcStages, or 2 when ksplit == 1 (two CTAs per SM)
  unsigned* counters;    // per M tile
  int n_mtiles;
  int* err;
};

__host__ __device__ inline size_t tc_stage_bytes(int bpad) {
  return 16384 /* raw weights (+scales) */ + 16384 /* A tile */ + (size_t)2 * bpad * 128 /* x parts */;
}
// The split-K merge (a 4-deep ring of [bpad/4][128] float4 partials) and the epilogue's two
// [bpad][128] float buffers reuse the stage buffers once the accumulator is complete: with a
// K split the ring and the buffers must fit in kTcStages stages, without one (2 stages, no
// ring) the buffers alone in 2, for every bpad up to 64.
static_assert(4 * 128 * 64 * 4 + 2 * 64 * 128 * 4 <= kTcStages * (16384 + 16384 + 2 * 64 * 128),
              "merge and epilogue buffers exceed the stage buffers");
static_assert(2 * 64 * 128 * 4 <= 2 * (16384 + 16384 + 2 * 16 * 128), "epilogue buffers exceed two stages");
__host__ __device__ inline size_t tc_smem_bytes(int bpad, int stages) {
  return 1024 /* alignment slack */ + stages * tc_stage_bytes(bpad) + 256 /* barriers, flags */;
}

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait that ignores the abort flag (draining copies / MMAs before teardown).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* b, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try(b, parity)) return true;
  return false;
}
// Bounded wait: false on expiry or when another role aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try(b, parity)) return true;
    if ((i & 1023) == 1023 && *abort_flag) return false;
  }
  return false;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
// K-major, 128-byte swizzle, 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                     // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;           // stride byte offset: next 8-row atom
  d |= (uint64_t)1 << 46;                     // descriptor version
  d |= (uint64_t)2 << 61;                     // 128-byte swizzle
  return d;
}
// kind::f16 instruction descriptor: bf16 A/B, fp32 D, both K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t umma_idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
}
// Byte offset of 16-byte chunk c (0..7) of row r in a swizzled [rows][64 bf16] tile.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kTcThreads, 1) gemm_tc_kernel(const GemmArgs a) {
  extern __shared__ __align__(16) uint8_t tc_raw_smem[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(tc_raw_smem) + 1023) & ~uintptr_t(1023));
  const size_t stage_bytes = tc_stage_bytes(a.bpad);
  uint8_t* stage0 = smem;
  const int NS = a.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NS * stage_bytes);
  uint64_t* full = bars;                     // [kTcStages] TMA data landed
  uint64_t* aready = bars + kTcStages;       // [kTcStages] dequantised tile written
  uint64_t* mdone = bars + 2 * kTcStages;    // [kTcStages] MMAs of the stage finished
  uint64_t* accdone = bars + 3 * kTcStages;  // accumulator complete
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 3 * kTcStages + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kTcStages + 2);
  int* is_last_s = reinterpret_cast<int*>(bars + 3 * kTcStages + 3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x / a.ksplit, ks = blockIdx.x % a.ksplit;
  const int kb0 = ks * a.kb_per_split;
  const int kb1 = min(a.n_kb, kb0 + a.kb_per_split);
  const int nkb = kb1 - kb0;
  const int ncols = a.bpad <= 32 ? 32 : (a.bpad <= 64 ? 64 : 128);

  // barriers, TMEM and the first stages' weights do not depend on the previous kernel: they
  // are set up and requested before the dependency wait (only the producer's activation
  // copies and the other warps' work come after it)
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&aready[s], 128);
      mbar_init(&mdone[s], 1);
    }
    mbar_init(accdone, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  const bool w4 = a.fmt == FMT_W4A16;
  const uint32_t xbytes = (uint32_t)a.bpad * 128;

  if (warp == 4) {
    // ---------------- TMA producer
    if (lane == 0) {
      int issued = 0;
      const uint32_t wbytes = w4 ? 4 * 1024 : 4 * 4096;
      const uint32_t sbytes = w4 ? 4 * 512 : 0;
      auto weights = [&](int i) {  // stage i's weight (and scale) copies
        const int s = i % NS;
        uint8_t* st = stage0 + s * stage_bytes;
        const int kb = kb0 + i;
        mbar_expect_tx(&full[s], wbytes + sbytes + 2 * xbytes);
        for (int rb = 0; rb < 4; ++rb) {
          const size_t grb = (size_t)mt * 4 + rb;
          if (w4) {
            const uint4* src = a.qw + (grb * a.tiles + (size_t)kb * 2) * 32;
            bulk_g2s(st + rb * 1024, src, 1024, &full[s]);
            const uint4* ssrc = a.sc + (grb * a.S + (kb >> 2)) * 32;
            bulk_g2s(st + 8192 + rb * 512, ssrc, 512, &full[s]);
          } else {
            const uint4* src = a.qw + (grb * a.tiles + (size_t)kb * 8) * 32;
            bulk_g2s(st + rb * 4096, src, 4096, &full[s]);
          }
        }
      };
      auto acts = [&](int i) {  // stage i's activation tiles (written by the previous kernel)
        const int s = i % NS;
        const uint8_t* xsrc = a.xt + (size_t)(kb0 + i) * 2 * xbytes;
        bulk_g2s(stage0 + s * stage_bytes + 32768, xsrc, 2 * xbytes, &full[s]);
      };
      const int npre = min(nkb, NS);
      for (int i = 0; i < npre; ++i) weights(i);
      pdl_wait();
      pdl_trigger();
      for (int i = 0; i < npre; ++i) acts(i);
      issued = npre;
      for (int i = npre; i < nkb; ++i) {
        const int s = i % NS, r = i / NS;
        if (r > 0 && !mbar_wait(&mdone[s], (r - 1) & 1, abort_flag)) {
          set_err(a.err, G4_DEV_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        weights(i);
        acts(i);
        ++issued;
      }
      if (*abort_flag) {
        // drain: every issued stage must land before the CTA exits
        for (int i = 0; i < issued; ++i) mbar_wait_drain(&full[i % NS], (i / NS) & 1);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer
    pdl_wait();
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(a.bpad);
      bool ok = true;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % NS, r = i / NS;
        if (!mbar_wait(&aready[s], r & 1, abort_flag)) { ok = false; break; }
        asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
        uint8_t* st = stage0 + s * stage_bytes;
        const uint32_t a_addr = su32(st + 16384);
        const uint32_t x_addr = su32(st + 32768);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint64_t ad = umma_desc_sw128(a_addr + kk * 32);
            const uint64_t bd = umma_desc_sw128(x_addr + part * xbytes + kk * 32);
            const uint32_t acc = (i > 0 || kk > 0 || part > 0) ? 1u : 0u;
            asm volatile(
                "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
                : "memory");
          }
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                         su32(&mdone[s]))
                     : "memory");
      }
      if (!ok) {
        set_err(a.err, G4_DEV_TIMEOUT);
        *abort_flag = 1;
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                       su32(accdone))
                   : "memory");
    }
  } else {
    // ---------------- dequant warps: thread m owns weight row m of the M tile
    pdl_wait();
    const int m = threadIdx.x;  // 0..127
    const int rbl = m >> 5, ln = m & 31;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % NS, r = i / NS;
      if (!mbar_wait(&full[s], r & 1, abort_flag)) {
        set_err(a.err, G4_DEV_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      uint8_t* st = stage0 + s * stage_bytes;
      uint8_t* A = st + 16384;
      const int kb = kb0 + i;
      if (w4) {
        const uint32_t sw = reinterpret_cast<const uint32_t*>(st + 8192 + rbl * 512 + ln * 16)[(kb & 3)];
        const __nv_bfloat162 bias = __floats2bfloat162_rn(136.f, 136.f);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint4 q = *reinterpret_cast<const uint4*>(st + rbl * 1024 + t * 512 + ln * 16);
          const uint32_t hh = t ? (sw >> 16) : (sw & 0xFFFFu);
          const __nv_bfloat162 sc = as_bf162(hh | (hh << 16));
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int mm = 0; mm < 4; ++mm) {
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t u = ((w[mm] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
              o[j] = as_u32(__hmul2(__hsub2(as_bf162(u), bias), sc));
            }
            const int c = t * 4 + mm;  // 16-byte chunk: k = 8c .. 8c+7 of the block
            *reinterpret_cast<uint4*>(A + sw128_off(m, c)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(st + rbl * 4096 + c * 512 + ln * 16);
          *reinterpret_cast<uint4*>(A + sw128_off(m, c)) = v;
        }
      }
      asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
      mbar_arrive(&aready[s]);
    }
    // ---------------- epilogue: wait for the accumulator, read TMEM row m
    const bool have = mbar_wait_drain(accdone, 0) && !*abort_flag;
    if (!have && m == 0) set_err(a.err, G4_DEV_TIMEOUT);
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    float v[64];
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 16) {
      if (c0 < a.bpad) {
        uint32_t r[16];
        const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0;
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
            "[%16];\n"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
        asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c0 + j] = __uint_as_float(r[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c0 + j] = 0.f;
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
    const int row = mt * kTcM + m;  // row of the tiled weight matrix
    const int rows_total = a.n_mtiles * kTcM;
    bool final_ok = have;
    if (a.ksplit > 1) {
      // partials [ksplit][row][64 columns]: each row's bpad columns are contiguous, so a thread
      // moves them as bpad / 4 float4 (written and read back with all loads of a split in flight)
      float4* prow = reinterpret_cast<float4*>(a.part) + ((size_t)ks * rows_total + row) * 16;
      if (have) {
#pragma unroll
        for (int c = 0; c < 16; ++c)
          if (4 * c < a.bpad) prow[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      }
      __threadfence();
      asm volatile("bar.sync 1, 128;\n" ::: "memory");
      if (m == 0) *is_last_s = atomicAdd(&a.counters[mt], 1u) == (unsigned)a.ksplit - 1;
      asm volatile("bar.sync 1, 128;\n" ::: "memory");
      final_ok = *is_last_s != 0;
      if (final_ok) {
        __threadfence();
#pragma unroll
        for (int b = 0; b < 64; ++b) v[b] = 0.f;
        // Each thread streams its row of every split's partial into its own slots of a 4-deep
        // shared ring with cp.async (up to 3 splits in flight), summing in split order.
        const int nc = a.bpad / 4;
        float4* qb = reinterpret_cast<float4*>(stage0);  // [4][nc][128 rows]
        auto issue = [&](int q) {
          const float4* pq = reinterpret_cast<const float4*>(a.part) + ((size_t)q * rows_total + row) * 16;
          float4* dst = qb + (size_t)(q & 3) * nc * kTcM;
          for (int c = 0; c < nc; ++c) cp_async16(dst + c * kTcM + m, pq + c, true);
          asm volatile("cp.async.commit_group;\n" ::: "memory");
        };
        for (int q = 0; q < 3 && q < a.ksplit; ++q) issue(q);
        for (int q = 0; q < a.ksplit; ++q) {
          if (q + 3 < a.ksplit) issue(q + 3);
          const int pending = min(a.ksplit, q + 4) - (q + 1);  // groups allowed to stay in flight
          if (pending >= 3) asm volatile("cp.async.wait_group 3;\n" ::: "memory");
          else if (pending == 2) asm volatile("cp.async.wait_group 2;\n" ::: "memory");
          else if (pending == 1) asm volatile("cp.async.wait_group 1;\n" ::: "memory");
          else asm volatile("cp.async.wait_group 0;\n" ::: "memory");
          const float4* src = qb + (size_t)(q & 3) * nc * kTcM;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c < nc) {
              const float4 t = src[c * kTcM + m];
              v[4 * c] += t.x;
              v[4 * c + 1] += t.y;
              v[4 * c + 2] += t.z;
              v[4 * c + 3] += t.w;
            }
          }
        }
        if (m == 0) a.counters[mt] = 0u;
      }
    }
    // Epilogue.  The tile's columns go to shared memory once ([b][128 rows], past the split-K
    // ring, which other threads may still be reading), and the variants below run as rolled
    // loops over b: fully unrolled 64-column epilogues ran once per CTA from a cold
    // instruction cache.  The stage buffers are idle once the accumulator is complete.
    float* ex = reinterpret_cast<float*>(stage0 + (a.ksplit > 1 ? (size_t)4 * kTcM * a.bpad * 4 : 0));  // [bpad][128]
    float* pl = ex + (size_t)a.bpad * kTcM;                                        // [bpad][128]
    if (final_ok) {
#pragma unroll
      for (int b = 0; b < 64; ++b)
        if (b < a.bpad) ex[b * kTcM + m] = v[b];
    }
    asm volatile("bar.sync 1, 128;\n" ::: "memory");  // every CTA of the split reaches it
    if (final_ok) {
      if (a.epi == EPI_GEGLU) {
        // rows interleave 32-row blocks: gate j, up j, gate j+1, up j+1 (warps 0..3)
        if ((warp & 1) == 0) {
          const int n = mt * 64 + (warp >> 1) * 32 + ln;
          if (n < a.n_valid)
            for (int b = 0; b < a.nb; ++b)
              a.y[(size_t)b * a.y_stride + n] = gelu_tanh(ex[b * kTcM + m]) * ex[b * kTcM + m + 32];
        }
      } else if (a.epi == EPI_ARGMAX) {
        // logits out; then per column b the max over the tile's 128 rows, warp w taking columns
        // w, w + 4, ...: one partial per (b, CTA)
        if (a.logits && row < a.n_valid)
          for (int b = 0; b < a.nb; ++b) a.logits[(size_t)b * a.logits_stride + row] = ex[b * kTcM + m];
        for (int b = warp; b < a.nb; b += 4) {
          float x = __int_as_float(0x7fc00000);
          int idx = 0x7fffffff;
#pragma unroll
          for (int j = 0; j < kTcM / 32; ++j) {
            const int r = ln + 32 * j;
            const float c = ex[b * kTcM + r];
            const int ci = mt * kTcM + r;
            if (ci < a.n_valid && argmax_better(c, ci, x, idx)) { x = c; idx = ci; }
          }
          warp_argmax(x, idx);
          if (ln == 0) {
            a.am_val[(size_t)b * gridDim.x + blockIdx.x] = x;
            a.am_idx[(size_t)b * gridDim.x + blockIdx.x] = idx;
          }
        }
      } else if (row < a.n_valid) {
        if (a.epi == EPI_PLE) {
          // the row's multipliers arrive by cp.async (one round trip, nothing waits on a
          // single load), [b][128 rows] so the accesses are conflict-free
          for (int b = 0; b < a.nb; ++b) cp_async4(pl + b * kTcM + m, a.ple + (size_t)b * a.ple_stride + row);
          cp_async_wait_all();
          for (int b = 0; b < a.nb; ++b)
            a.y[(size_t)b * a.y_stride + row] = gelu_tanh(ex[b * kTcM + m]) * pl[b * kTcM + m];
        } else {
          for (int b = 0; b < a.nb; ++b) a.y[(size_t)b * a.y_stride + row] = ex[b * kTcM + m];
        }
      }
    }
  }
  __syncthreads();
  if (warp == 4) {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(ncols) : "memory");
  }
}

// Activation tiles for the tensor-core GEMM: the GEMV prologue (plain / RMSNorm / residual
// update + RMSNorm) per row, then x_hi = bf16(x) and x_lo = bf16(x - x_hi) written as
// 128-byte-swizzled [bpad rows][64 k] tiles, tile (kb, part) at byte (kb * 2 + part) *
// bpad * 128.  One CTA per activation row; rows >= nb are left as they are (their GEMM
// columns are never read).
struct PrepArgs {
  int pro;
  const float* x_in;
  int x_stride;
  const float* r_in;
  int r_stride;
  const __nv_bfloat16* g_r;
  float lambda;
  const __nv_bfloat16* g_a;
  float* x_out;
  float eps;
  int K;          // logical activation length
  int kpad;       // n_kb * 64
  int bpad;
  uint8_t* xt;
};

// Shared memory of prep_x_kernel: x row and residual branch (fp32, kpad each), then both gain
// vectors (bf16, kpad each).
__host__ __device__ inline size_t prep_smem_bytes(int kpad, int pro) {
  return pro == PRO_PLAIN ? (size_t)kpad * 4 : (size_t)kpad * (2 * 4 + 2 * 2);  // plain: the x row only
}

__global__ void __launch_bounds__(256) prep_x_kernel(const PrepArgs a) {
  extern __shared__ __align__(16) float prow[];  // [kpad] | residual [kpad] | g_r, g_a [kpad] bf16
  __shared__ float red[32];
  const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  float* rrow = prow + a.kpad;
  __nv_bfloat16* gr_s = reinterpret_cast<__nv_bfloat16*>(rrow + a.kpad);
  __nv_bfloat16* ga_s = gr_s + a.kpad;
  const bool resid = a.pro == PRO_RESID, norm = a.pro != PRO_PLAIN && a.g_a != nullptr;
  // gains are weights: staged before waiting for the previous kernel
  for (int c = tid; c < a.K / 8; c += nt) {
    if (resid) cp_async16(gr_s + 8 * c, a.g_r + 8 * c, true);
    if (norm) cp_async16(ga_s + 8 * c, a.g_a + 8 * c, true);
  }
  pdl_wait();
  pdl_trigger();
  const float* x = a.x_in + (size_t)b * a.x_stride;
  for (int c = tid; c < a.kpad / 4; c += nt) {
    const bool ok = 4 * c < a.K;
    cp_async16(prow + 4 * c, ok ? x + 4 * c : x, ok);
    if (resid && ok) cp_async16(rrow + 4 * c, a.r_in + (size_t)b * a.r_stride + 4 * c, true);
  }
  cp_async_wait_all();
  __syncthreads();
  // the loops below read only shared memory
  if (resid) {
    const float* r = rrow;
    float ss[1] = {0.f};
    for (int k = tid; k < a.K; k += nt) ss[0] += r[k] * r[k];
    block_sum<1>(ss, red);
    const float rd = rms_denom(ss[0], a.K, a.eps), lambda = a.lambda;
    for (int k = tid; k < a.K; k += nt) prow[k] = (prow[k] + (r[k] / rd) * bf16f(gr_s[k])) * lambda;
    __syncthreads();
    float* xo = a.x_out + (size_t)b * a.x_stride;
    for (int c = tid; c < a.K / 4; c += nt) reinterpret_cast<float4*>(xo)[c] = reinterpret_cast<const float4*>(prow)[c];
  }
  if (norm) {
    float ss[1] = {0.f};
    for (int k = tid; k < a.K; k += nt) ss[0] += prow[k] * prow[k];
    block_sum<1>(ss, red);
    const float ad = rms_denom(ss[0], a.K, a.eps);
    for (int k = tid; k < a.K; k += nt) prow[k] = (prow[k] / ad) * bf16f(ga_s[k]);
    __syncthreads();
  }
  const size_t tile = (size_t)a.bpad * 128;
  for (int c = tid; c < a.kpad / 8; c += nt) {  // one 16-byte chunk (8 k) per iteration
    const int kb = c >> 3, ci = c & 7;
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v0 = prow[c * 8 + 2 * j], v1 = prow[c * 8 + 2 * j + 1];
      const __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(v0 - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(v1 - __bfloat162float(h1));
      hi[j] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      lo[j] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
    }
    uint8_t* base = a.xt + (size_t)kb * 2 * tile + sw128_off(b, ci);
    *reinterpret_cast<uint4*>(base) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(base + tile) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// Final argmax over per-CTA partials: one block per activation row.
__global__ void argmax_partials_kernel(const float* pv, const int* pi, int n_part, int* ids) {
  __shared__ float sv[32];
  __shared__ int si[32];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float v = __int_as_float(0x7fc00000);
  int idx = 0x7fffffff;
  for (int c = threadIdx.x; c < n_part; c += blockDim.x) {
    const float x = pv[(size_t)b * n_part + c];
    const int xi = pi[(size_t)b * n_part + c];
    if (argmax_better(x, xi, v, idx)) { v = x; idx = xi; }
  }
  warp_argmax(v, idx);
  if (lane == 0) { sv[warp] = v; si[warp] = idx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < nw; ++w)
      if (argmax_better(sv[w], si[w], sv[0], si[0])) { sv[0] = sv[w]; si[0] = si[w]; }
    ids[b] = si[0] == 0x7fffffff ? 0 : si[0];
  }
}

}  // namespace g4
