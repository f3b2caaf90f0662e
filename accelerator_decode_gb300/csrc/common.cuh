// Shared device helpers for libg4 (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/g4.h"

namespace g4 {

constexpr int kWarp = 32;

// ---------------------------------------------------------------------------- bf16 helpers
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t u) {
  return *reinterpret_cast<__nv_bfloat162*>(&u);
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}

// ----------------------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// (value, index) argmax: larger value wins; equal values -> lower index; NaN never wins.
__device__ __forceinline__ bool argmax_better(float v, int i, float bv, int bi) {
  if (v != v) return false;
  if (bv != bv) return true;
  return v > bv || (v == bv && i < bi);
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    int oi = __shfl_xor_sync(0xFFFFFFFFu, i, o);
    if (argmax_better(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

// Sum of NB values over the block (blockDim.x a multiple of 32, <= 1024).  `red` must hold
// 32 * NB floats.  Every thread gets the totals.
template <int NB>
__device__ __forceinline__ void block_sum(float (&v)[NB], float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int b = 0; b < NB; ++b) v[b] = warp_sum(v[b]);
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int b = 0; b < NB; ++b) red[b * 32 + warp] = v[b];
  }
  __syncthreads();
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[b * 32 + w];
    v[b] = s;
  }
  __syncthreads();
}

// tanh-form GELU, same expression order as the oracle.
__device__ __forceinline__ float gelu_tanh(float z) {
  const float c = 0.7978845608028654f;  // sqrt(2/pi) rounded to fp32
  return 0.5f * z * (1.0f + tanhf(c * (z + 0.044715f * z * z * z)));
}

// RMSNorm scale: 1 / sqrt(mean + eps) is applied as a division, v / sqrt(ss/n + eps).
__device__ __forceinline__ float rms_denom(float ss, int n, float eps) {
  return sqrtf(ss / (float)n + eps);
}

__device__ __forceinline__ void set_err(int* err, int bit) {
  if (err) atomicOr(err, bit);
}

// Loads that bypass L1 (data written by other CTAs of the same grid).
__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }

// 16-byte global -> shared async copy; with pred == false the 16 bytes are zero-filled and
// nothing is read (src must still be a valid address).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool pred) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  const int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(sz) : "memory");
}
// 4-byte global -> shared async copy (through L1; both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Programmatic dependent launch.  Before pdl_wait() a kernel may only read data that no
// kernel of the step writes (weights, RoPE tables); every global write and every read of an
// activation comes after it.  Kernels trigger their dependents only after their own wait, so
// at most two kernels of the step are resident at once (the one computing and the next one
// loading its weights): triggered at the start, every following kernel became resident in a
// cascade, SMs ran out of room, and the CTA scheduler put two CTAs of one kernel on one SM
// (half speed) while other SMs had none.  Both are no-ops for a launch without the PDL
// attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

}  // namespace g4
