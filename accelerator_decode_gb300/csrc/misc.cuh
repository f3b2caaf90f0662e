// Embedding gather, per-layer-embedding combine, weight repacking, standalone argmax.
#pragma once
#include "common.cuh"

namespace g4 {

// x0[b] = E[t_b] * sqrt(H);  tok[b] = T_ple[t_b] * sqrt(P)   (fp32)
// Token ids come from tokens[b] or, with idx != nullptr, tokens[idx[b]].
// "Porting Gemma 4 E2B to SGLang-JAX", Step 3: tok = embed_tokens_per_layer(ids) * ple_dim**0.5.
// int4 tables ("Six serving engines on one Cloud TPU v5e chip", What Changes and What Stays):
// rows of packed int32 words (8 signed nibbles, low first) with a bf16 scale per `group`
// values; a table value is bf16(q * s) as for the int4 linears.
struct EmbedArgs {
  const int* tokens;
  const int* idx;
  const __nv_bfloat16* embed;      // [V][H] (bf16 tables)
  const __nv_bfloat16* ple_table;  // [V][LP]
  int V, H, LP;
  float sqrt_h, sqrt_p;
  float* x0;   // [nb][H]
  float* tok;  // [nb][LP]
  int* err;
  // int4 tables (t4): words [V][H/8] / [V][LP/8], scales [V][H/32] / [V][LP/ple_group]
  int t4;
  const uint32_t* embed_q;
  const __nv_bfloat16* embed_s;
  const uint32_t* ple_q;
  const __nv_bfloat16* ple_s;
  int ple_group;
};

// Grid (ceil((H + LP) / (8 * blockDim.x)), nb): each thread converts 8 bf16 (one 16-byte load).
__global__ void embed_kernel(const EmbedArgs a) {
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y;
  int t = a.idx ? a.tokens[a.idx[b]] : a.tokens[b];
  if (t < 0 || t >= a.V) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_err(a.err, G4_DEV_BAD_TOKEN);
    t = 0;
  }
  const int i8 = (blockIdx.x * blockDim.x + threadIdx.x) * 8;  // element index over [x0 | tok]
  const __nv_bfloat16* src;
  float* dst;
  float sc;
  if (i8 < a.H) {
    src = a.embed + (size_t)t * a.H + i8;
    dst = a.x0 + (size_t)b * a.H + i8;
    sc = a.sqrt_h;
  } else if (i8 < a.H + a.LP) {
    src = a.ple_table + (size_t)t * a.LP + (i8 - a.H);
    dst = a.tok + (size_t)b * a.LP + (i8 - a.H);
    sc = a.sqrt_p;
  } else {
    return;
  }
  if (a.t4) {  // one word of 8 nibbles; a scale group holds whole words
    const bool e = i8 < a.H;
    const int k = e ? i8 : i8 - a.H;
    const uint32_t w = e ? a.embed_q[(size_t)t * (a.H / 8) + k / 8] : a.ple_q[(size_t)t * (a.LP / 8) + k / 8];
    const float s = e ? bf16f(a.embed_s[(size_t)t * (a.H / 32) + k / 32])
                      : bf16f(a.ple_s[(size_t)t * (a.LP / a.ple_group) + k / a.ple_group]);
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = (int)((w >> (4 * j)) & 0xFu) - (((w >> (4 * j)) & 0x8u) ? 16 : 0);
      v[j] = bf16f(__float2bfloat16_rn((float)q * s)) * sc;  // q * s is exact in fp32
    }
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
    return;
  }
  const uint4 u = *reinterpret_cast<const uint4*>(src);
  const float4 lo = make_float4(bf16_lo(u.x) * sc, bf16_hi(u.x) * sc, bf16_lo(u.y) * sc, bf16_hi(u.y) * sc);
  const float4 hi = make_float4(bf16_lo(u.z) * sc, bf16_hi(u.z) * sc, bf16_lo(u.w) * sc, bf16_hi(u.w) * sc);
  reinterpret_cast<float4*>(dst)[0] = lo;
  reinterpret_cast<float4*>(dst)[1] = hi;
}

// ple[b][l] = (RMSNorm(pr[b][l] * H^-1/2) * g + tok[b][l]) * 2^-1/2, one block per (b, l).
// "Porting Gemma 4 E2B to SGLang-JAX", Step 3 (per-layer projection norm and the combine).
// pr may come as `parts` K-slice partial sums (part q at pr + q * part_stride), added in order.
__global__ void ple_combine_kernel(const float* pr, int parts, long part_stride, const float* tok,
                                   const __nv_bfloat16* g, int L, int P, float inv_sqrt_h, float inv_sqrt2, float eps,
                                   float* ple) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y, l = blockIdx.x;
  const size_t base = ((size_t)b * L + l) * P;
  float ss[1] = {0.f};
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    float v = __ldcg(pr + base + i);
    for (int q = 1; q < parts; ++q) v += __ldcg(pr + q * part_stride + base + i);
    v *= inv_sqrt_h;
    ss[0] += v * v;
  }
  block_sum<1>(ss, red);
  const float den = rms_denom(ss[0], P, eps);
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    float v = __ldcg(pr + base + i);
    for (int q = 1; q < parts; ++q) v += __ldcg(pr + q * part_stride + base + i);
    v *= inv_sqrt_h;
    ple[base + i] = ((v / den) * bf16f(g[i]) + tok[base + i]) * inv_sqrt2;
  }
}

// Row gather for prefill blocks: dst row i = src row idx[i] (width floats, a multiple of 4;
// strides in floats, multiples of 4).  dst and src must not overlap.
__global__ void gather_rows_kernel(const float* src, int src_stride, float* dst, int dst_stride, const int* idx,
                                   int width) {
  pdl_wait();
  pdl_trigger();
  const int i = blockIdx.x;
  const float4* s4 = reinterpret_cast<const float4*>(src + (size_t)__ldcg(idx + i) * src_stride);
  float4* d4 = reinterpret_cast<float4*>(dst + (size_t)i * dst_stride);
  for (int c = threadIdx.x; c < width / 4; c += blockDim.x) d4[c] = __ldcg(s4 + c);
}

// ------------------------------------------------------------------------------ repacking
// One destination 32-row block: `w` points at its first source row (nullptr = zero block),
// `s` at its first scale row (W4A16), `rows` valid rows (<= 32).
struct RbSrc {
  const void* w;
  const void* s;
  int rows;
  int pad;
};

// Canonical int4 (k at word k/8, bits 4*(k%8), two's complement) -> tiled offset-binary.
__global__ void repack_int4_kernel(const RbSrc* srcs, int n_rb, int K, int tiles, uint4* qw) {
  const size_t total = (size_t)n_rb * tiles * 32;
  const int G = K / 32;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int lane = i % 32;
    const int g = (i / 32) % tiles;
    const int rb = i / (32 * (size_t)tiles);
    const RbSrc s = srcs[rb];
    uint32_t out[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};  // q = 0
    if (s.w != nullptr && lane < s.rows && g < G) {
      const uint32_t* row = reinterpret_cast<const uint32_t*>(s.w) + (size_t)lane * (K / 8);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t c = row[4 * g + m];
        uint32_t o = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t nib = ((c >> (4 * e)) & 0xFu) ^ 0x8u;
          const int pos = (e & 1) ? 16 + 4 * (e >> 1) : 4 * (e >> 1);
          o |= nib << pos;
        }
        out[m] = o;
      }
    }
    qw[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// bf16 scales [N][K/32] -> sc[(rb * S + sg) * 32 + lane] = 8 scales of groups 8sg..8sg+7.
__global__ void repack_scales_kernel(const RbSrc* srcs, int n_rb, int K, int S, uint4* sc) {
  const size_t total = (size_t)n_rb * S * 32;
  const int G = K / 32;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int lane = i % 32;
    const int sg = (i / 32) % S;
    const int rb = i / (32 * (size_t)S);
    const RbSrc s = srcs[rb];
    uint16_t v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int g = sg * 8 + t;
      v[t] = 0;
      if (s.s != nullptr && lane < s.rows && g < G)
        v[t] = reinterpret_cast<const uint16_t*>(s.s)[(size_t)lane * G + g];
    }
    sc[i] = make_uint4(v[0] | (uint32_t(v[1]) << 16), v[2] | (uint32_t(v[3]) << 16),
                       v[4] | (uint32_t(v[5]) << 16), v[6] | (uint32_t(v[7]) << 16));
  }
}

// bf16 row-major [N][K] -> tiled: qw[(rb * tiles + c) * 32 + lane] = row k in [8c, 8c+8).
__global__ void repack_bf16_kernel(const RbSrc* srcs, int n_rb, int K, int tiles, uint4* qw) {
  const size_t total = (size_t)n_rb * tiles * 32;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int lane = i % 32;
    const int c = (i / 32) % tiles;
    const int rb = i / (32 * (size_t)tiles);
    const RbSrc s = srcs[rb];
    uint4 out = make_uint4(0, 0, 0, 0);
    if (s.w != nullptr && lane < s.rows && 8 * c < K)
      out = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(s.w) + (size_t)lane * K + 8 * c);
    qw[i] = out;
  }
}

// ------------------------------------------------------------------------ standalone argmax
// Block partials over column chunks, then the last block reduces (same scheme as the lm_head).
__global__ void argmax_rows_kernel(const float* logits, int n_cols, int chunk, float* pv, int* pi,
                                   unsigned* counter, int* ids) {
  const int row = blockIdx.y, c = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __shared__ float sv[32];
  __shared__ int si[32];
  float v = __int_as_float(0x7fc00000);
  int idx = 0x7fffffff;
  const int c0 = c * chunk, c1 = min(n_cols, c0 + chunk);
  for (int j = c0 + threadIdx.x; j < c1; j += blockDim.x) {
    const float x = logits[(size_t)row * n_cols + j];
    if (argmax_better(x, j, v, idx)) { v = x; idx = j; }
  }
  warp_argmax(v, idx);
  if (lane == 0) { sv[warp] = v; si[warp] = idx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < nw; ++w)
      if (argmax_better(sv[w], si[w], sv[0], si[0])) { sv[0] = sv[w]; si[0] = si[w]; }
    pv[row * gridDim.x + c] = sv[0];
    pi[row * gridDim.x + c] = si[0];
  }
  __threadfence();
  __syncthreads();
  __shared__ int is_last;
  if (threadIdx.x == 0) is_last = atomicAdd(&counter[row], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  v = __int_as_float(0x7fc00000);
  idx = 0x7fffffff;
  for (int j = threadIdx.x; j < (int)gridDim.x; j += blockDim.x) {
    const float x = ldcg(pv + row * gridDim.x + j);
    const int xi = __ldcg(pi + row * gridDim.x + j);
    if (argmax_better(x, xi, v, idx)) { v = x; idx = xi; }
  }
  warp_argmax(v, idx);
  __syncthreads();
  if (lane == 0) { sv[warp] = v; si[warp] = idx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < nw; ++w)
      if (argmax_better(sv[w], si[w], sv[0], si[0])) { sv[0] = sv[w]; si[0] = si[w]; }
    ids[row] = si[0] == 0x7fffffff ? 0 : si[0];
    counter[row] = 0u;
  }
}

// Failure-detection probe: one warp waits for *flag to become non-zero, checking
// %globaltimer, and gives up after wait_ns: the timeout bit goes to the error word and the
// kernel returns (the wait always ends; the context stays usable).  Nothing sets the flag
// the library passes, so the probe exercises the bounded-wait path of the step's kernels.
__global__ void probe_wait_kernel(const int* flag, unsigned long long wait_ns, int* err) {
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  for (;;) {
    if (*reinterpret_cast<const volatile int*>(flag) != 0) return;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > wait_ns) break;
    __nanosleep(1000);
  }
  if (threadIdx.x == 0) set_err(err, G4_DEV_TIMEOUT);
}

}  // namespace g4
