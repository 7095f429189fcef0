// Shared device helpers for the gdnbeam kernels: storage-type traits, the
// device error word, and launch error plumbing.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/gdnbeam.h"

namespace gdnbeam {

// Kernels receive the address of the device error word and OR
// GDNBEAM_DERR_* bits into it, skipping the offending access instead of
// trapping.
__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// ---- storage types -------------------------------------------------------

template <typename T> struct St;
template <> struct St<float> {
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
  static constexpr int kDtype = GDNBEAM_F32;
};
template <> struct St<__nv_bfloat16> {
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  static constexpr int kDtype = GDNBEAM_BF16;
};

template <typename T> __device__ __forceinline__ float ldf(const T* p) { return St<T>::load(p); }
template <typename T> __device__ __forceinline__ void stf(T* p, float x) { *p = St<T>::from_f(x); }

// Gates (OneLA §1.2 eq. 3 inputs): alpha = exp(-softplus(z)) is evaluated
// as the logistic function at -z, which is the same value; beta = sigmoid(z).
__device__ __forceinline__ float decay_gate(float z) { return 1.0f / (1.0f + expf(z)); }
__device__ __forceinline__ float write_gate(float z) { return 1.0f / (1.0f + expf(-z)); }

// Orderable 32-bit image of an fp32 score (larger float -> larger integer).
// -0 and +0 map to the same image.
__device__ __forceinline__ uint32_t orderable(float s) {
  if (s == 0.0f) s = 0.0f;  // -0 -> +0
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_orderable(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(u);
}

}  // namespace gdnbeam

namespace gdnbeam {
// Counts kernel launches issued by the library (defined in api.cu).
void note_launch();
}  // namespace gdnbeam

// Host-side launch checking; every kernel launch is followed by this.
#define GDN_LAUNCH_CHECK()                                 \
  do {                                                     \
    gdnbeam::note_launch();                                \
    cudaError_t e_ = cudaGetLastError();                   \
    if (e_ != cudaSuccess) return GDNBEAM_ECUDA;           \
  } while (0)

#define GDN_CUDA(call)                                     \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return GDNBEAM_ECUDA;           \
  } while (0)
