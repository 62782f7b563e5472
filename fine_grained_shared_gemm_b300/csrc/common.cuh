// Device helpers shared by the kernels of the MoE layer forward (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Bits of the per-device error word.  Kernels set a bit instead of trapping
// when a bounded wait expires or an index is out of range.
enum : int {
  DEV_ERR_TIMEOUT_PRODUCER = 1,
  DEV_ERR_TIMEOUT_MMA = 2,
  DEV_ERR_TIMEOUT_EPILOGUE = 4,
  DEV_ERR_BAD_EXPERT = 8,
  DEV_ERR_SMEM_SHORT = 16,  // launched with less dynamic shared memory than its layout
};

// Upper bound on any single wait inside a kernel (nanoseconds of the global
// timer).  No wait in a correct launch comes near it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ int g_device_error;

__device__ __forceinline__ void raise_device_error(int bits) {
  atomicOr(&g_device_error, bits);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_float(float x);
template <> __device__ __forceinline__ float from_float<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const float* p, float* v) {
    float4 q = *reinterpret_cast<const float4*>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
  __device__ static void store(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
};
template <> struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void load(const __nv_bfloat16* p, float* v) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x; v[2 * i + 1] = f.y;
    }
  }
  __device__ static void store(__nv_bfloat16* p, const float* v) {
    uint4 q;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = q;
  }
};

// One expert group of a grouped GEMM: which weight stack and token source it
// reads, where its rows start and how many token rows it has.
struct GroupDesc {
  int a_sel;     // 0 = routed weight stack, 1 = shared weight stack
  int a_row0;    // first weight row of this expert in its stack
  int b_src;     // token source: 0 or 1 (meaning depends on the GEMM)
  int b_row0;    // first token row in that source
  int out_sel;   // output buffer: 0 or 1
  int out_row0;  // first output row
  int count;     // token rows
  int pad;
};

}  // namespace moe
