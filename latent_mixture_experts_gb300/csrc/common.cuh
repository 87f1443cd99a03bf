// Device helpers shared by the layer's kernels: activations, number formats,
// block scaling of activations into two E4M3 terms.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cstdint>

#include "ptx.cuh"

namespace lmoe {

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ float sigmoidf_(float z) { return 1.0f / (1.0f + expf(-z)); }

// SiTU-GLU (Kimi K3 card, routed-expert steps): a = b1 tanh(g/b1) sigma(g),
// u_bar = b2 tanh(u/b2), h = a * u_bar.  act == 1: SwiGLU g sigma(g) u
// (Kimi K2 card, routed-expert steps).
__device__ __forceinline__ float glu_act(float g, float u, int act, float b1, float b2) {
  if (act == 1) return g * sigmoidf_(g) * u;
  const float a = b1 * tanhf(g / b1) * sigmoidf_(g);
  const float ub = b2 * tanhf(u / b2);
  return a * ub;
}

// Hardware approximations for the expert epilogues, whose output is encoded
// as E4M3 terms right after (relative error ~2^-11: below the resolution of
// two terms; with one term it moves about one value in a hundred to the
// adjacent code, a choice as valid as the rounding of the exact value).
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sigmoid_fast(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }
__device__ __forceinline__ float glu_act_fast(float g, float u, int act, float b1, float b2) {
  const float sg = sigmoid_fast(g);
  if (act == 1) return g * sg * u;
  return b1 * tanh_fast(g * (1.0f / b1)) * sg * (b2 * tanh_fast(u * (1.0f / b2)));
}

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t q) {
  __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(q), __NV_E4M3);
  return __half2float(__half(h));
}
// 2^(e - 127) for an E8M0 byte e in [1, 254], built from its bit pattern.
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) { return __uint_as_float(e << 23); }

// E8M0 scale byte for a 32-element block whose largest magnitude is amax:
// the smallest power of two with amax / scale <= 448, the largest finite
// E4M3.  With s = exponent(amax) - 8, amax / scale = 256 * (1 + mantissa),
// which passes 448 once the mantissa exceeds 0.75; such a block takes the
// next scale up (amax / scale in (224, 256]) so that no code saturates —
// a saturated hi code leaves a residual the lo term, scaled the same way,
// cannot hold either.  Clamped so the scale and its reciprocal stay normal.
__device__ __forceinline__ uint32_t e4m3_block_scale(float amax) {
  const uint32_t bits = __float_as_uint(amax);
  const int ef = static_cast<int>((bits >> 23) & 0xFF);
  int s = ef - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  s = s < 1 ? 1 : (s > 253 ? 253 : s);
  return static_cast<uint32_t>(s);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
// Largest of 32 non-negative values (one per lane), all lanes: the bit
// patterns of non-negative floats order as unsigned integers, so one
// warp-wide integer max reduction gives the float maximum exactly.
__device__ __forceinline__ float warp_amax(float nonneg) {
  return __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(nonneg)));
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Two-term E4M3 encoding of one element of a 32-element block held across
// the 32 lanes of a warp: a ~= q_hi * 2^(s_hi-127) + q_lo * 2^(s_lo-127),
// the second term quantising the first one's exact residual with its own
// block scale.  Every lane gets its codes; all lanes get the two scales.
struct HiLo {
  uint8_t q_hi, q_lo;
  uint32_t s_hi, s_lo;
};
__device__ __forceinline__ HiLo quant_hilo_warp(float a) {
  HiLo r;
  const float amax = warp_amax(fabsf(a));
  r.s_hi = e4m3_block_scale(amax);
  r.q_hi = f32_to_e4m3(a * e8m0_to_f32(254u - r.s_hi));
  const float res = a - e4m3_to_f32(r.q_hi) * e8m0_to_f32(r.s_hi);
  const float rmax = warp_amax(fabsf(res));
  r.s_lo = e4m3_block_scale(rmax);
  r.q_lo = f32_to_e4m3(res * e8m0_to_f32(254u - r.s_lo));
  return r;
}

// quant_hilo_warp on N independent values per lane (N tokens of the same
// 32-block): the N warp reductions run interleaved, so their shuffle
// latencies overlap.  Same result as N calls of quant_hilo_warp.
template <int N>
__device__ __forceinline__ void quant_hilo_warp_n(const float (&a)[N], HiLo (&r)[N]) {
  float m[N], res[N];
#pragma unroll
  for (int u = 0; u < N; ++u) m[u] = fabsf(a[u]);
#pragma unroll
  for (int u = 0; u < N; ++u) m[u] = warp_amax(m[u]);
#pragma unroll
  for (int u = 0; u < N; ++u) {
    r[u].s_hi = e4m3_block_scale(m[u]);
    r[u].q_hi = f32_to_e4m3(a[u] * e8m0_to_f32(254u - r[u].s_hi));
    res[u] = a[u] - e4m3_to_f32(r[u].q_hi) * e8m0_to_f32(r[u].s_hi);
    m[u] = fabsf(res[u]);
  }
#pragma unroll
  for (int u = 0; u < N; ++u) m[u] = warp_amax(m[u]);
#pragma unroll
  for (int u = 0; u < N; ++u) {
    r[u].s_lo = e4m3_block_scale(m[u]);
    r[u].q_lo = f32_to_e4m3(res[u] * e8m0_to_f32(254u - r[u].s_lo));
  }
}

// One-term form (MXFP8 activations): each value as a single E4M3 code with
// its block's scale; the lo term is an exact zero (code 0, scale 1) so that
// layouts holding a lo slot add nothing for it.
template <int N>
__device__ __forceinline__ void quant_hi_warp_n(const float (&a)[N], HiLo (&r)[N]) {
  float m[N];
#pragma unroll
  for (int u = 0; u < N; ++u) m[u] = fabsf(a[u]);
#pragma unroll
  for (int u = 0; u < N; ++u) m[u] = warp_amax(m[u]);
#pragma unroll
  for (int u = 0; u < N; ++u) {
    r[u].s_hi = e4m3_block_scale(m[u]);
    r[u].q_hi = f32_to_e4m3(a[u] * e8m0_to_f32(254u - r[u].s_hi));
    r[u].q_lo = 0;
    r[u].s_lo = 127u;
  }
}
// The encoding of h for the down pass: two terms, or one (terms == 1).
template <int N>
__device__ __forceinline__ void quant_terms_warp_n(const float (&a)[N], HiLo (&r)[N], int terms) {
  if (terms == 1)
    quant_hi_warp_n<N>(a, r);
  else
    quant_hilo_warp_n<N>(a, r);
}

// Programmatic dependent launch: the kernels of a forward are launched with
// programmatic stream serialization, so a kernel's CTAs may start while its
// predecessor drains.  Each kernel lets its successor launch at once and,
// before its first global read or write, waits until the predecessor grid
// has completed and its memory is visible (a no-op without the attribute).
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Byte offset of one scale inside the tensor-memory staging image of a
// 128-row (or 128-column) operand block: 32 lines of 16 bytes, line r0 holds
// for c = 0..3 the four k-block scales of row 32c + r0.  This is the image
// tcgen05.cp.32x128b.warpx4 replicates into the four lane quarters, where
// the block-scaled MMA reads row n at lane n % 32, column n / 32, byte =
// the k-block's scale id.
__device__ __forceinline__ uint32_t sf_atom_offset(uint32_t n_in_128, uint32_t kb_in_4) {
  return (n_in_128 & 31u) * 16u + (n_in_128 >> 5) * 4u + kb_in_4;
}

}  // namespace lmoe
