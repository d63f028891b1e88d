// Device helpers shared by the on-chip tensor-core kernels (ns_tc.cu, ns_pair.cu):
// the 128-byte-swizzled bf16 / fp32 tile layouts of their shared-memory operands,
// packed fp32 pair arithmetic, 32-element row segments of global matrices, and
// bounded mbarrier waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace himuon {
namespace tile {

// ------------------------------------------------------------------ layouts
// bf16 tile: element (r, c) in block c / 64, 16-byte chunk ((c % 64) / 8) ^ (r % 8).
__device__ __forceinline__ uint32_t bf_off(int r, int c8) {   // c8 = c / 8
  return static_cast<uint32_t>((c8 >> 3) * 16384 + r * 128 + (((c8 & 7) ^ (r & 7)) << 4));
}
// fp32 tile: element (r, c) in block c / 32, 16-byte chunk ((c % 32) / 4) ^ (r % 8).
__device__ __forceinline__ uint32_t f32_off(int r, int c4) {  // c4 = c / 4
  return static_cast<uint32_t>((c4 >> 3) * 16384 + r * 128 + (((c4 & 7) ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ packed fp32 pairs
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// v[j] *= s for 32 values, in pairs
__device__ __forceinline__ void scale32(float (&v)[32], float s) {
  const uint64_t ss = pk2(s, s);
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    uint64_t x = mul2(pk2(v[j], v[j + 1]), ss);
    upk2(x, v[j], v[j + 1]);
  }
}

// 32 fp32 -> 16 packed bf16x2 -> 4 x 16-byte chunks of a bf16 tile row
__device__ __forceinline__ void st_bf16_32(uint32_t tile, int r, int c, const float (&v)[32],
                                           uint32_t (&pkd)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) pkd[j] = ptx::pack_bf16x2(v[2 * j], v[2 * j + 1]);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    ptx::st_shared_v4(tile + bf_off(r, (c >> 3) + q), pkd[4 * q], pkd[4 * q + 1], pkd[4 * q + 2],
                      pkd[4 * q + 3]);
}

__device__ __forceinline__ void ld_bf16_32(uint32_t tile, int r, int c, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u = ptx::ld_shared_v4(tile + bf_off(r, (c >> 3) + q));
    v[8 * q + 0] = ptx::bf16lo(u.x); v[8 * q + 1] = ptx::bf16hi(u.x);
    v[8 * q + 2] = ptx::bf16lo(u.y); v[8 * q + 3] = ptx::bf16hi(u.y);
    v[8 * q + 4] = ptx::bf16lo(u.z); v[8 * q + 5] = ptx::bf16hi(u.z);
    v[8 * q + 6] = ptx::bf16lo(u.w); v[8 * q + 7] = ptx::bf16hi(u.w);
  }
}

__device__ __forceinline__ void ld_f32_32(uint32_t tile, int r, int c, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint4 u = ptx::ld_shared_v4(tile + f32_off(r, (c >> 2) + q));
    v[4 * q + 0] = __uint_as_float(u.x); v[4 * q + 1] = __uint_as_float(u.y);
    v[4 * q + 2] = __uint_as_float(u.z); v[4 * q + 3] = __uint_as_float(u.w);
  }
}

__device__ __forceinline__ void st_f32_32(uint32_t tile, int r, int c, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    ptx::st_shared_v4(tile + f32_off(r, (c >> 2) + q), __float_as_uint(v[4 * q]),
                      __float_as_uint(v[4 * q + 1]), __float_as_uint(v[4 * q + 2]),
                      __float_as_uint(v[4 * q + 3]));
}

// single elements of the staging tiles (for tiles processed transposed)
__device__ __forceinline__ float f32_at(uint32_t tile, int r, int c) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(tile + f32_off(r, c >> 2) + (c & 3) * 4));
  return v;
}
__device__ __forceinline__ float bf16_at(uint32_t tile, int r, int c) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(tile + bf_off(r, c >> 3) + (c & 7) * 2));
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}

__device__ __forceinline__ void f32_put(uint32_t tile, int r, int c, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(tile + f32_off(r, c >> 2) + (c & 3) * 4), "f"(v) : "memory");
}

// ------------------------------------------------------------------ global row segments
// 32 elements from column c0 of a row, n of them valid (0..32); vector access
// when all 32 are valid and the row allows 16-byte access.
__device__ __forceinline__ void gload32(const void* rowp, int c0, int n, bool fp32, bool vec,
                                        float (&v)[32]) {
  if (n >= 32 && vec) {
    if (fp32) {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 f = p[q];
        v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
      }
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = p[q];
        v[8 * q + 0] = ptx::bf16lo(u.x); v[8 * q + 1] = ptx::bf16hi(u.x);
        v[8 * q + 2] = ptx::bf16lo(u.y); v[8 * q + 3] = ptx::bf16hi(u.y);
        v[8 * q + 4] = ptx::bf16lo(u.z); v[8 * q + 5] = ptx::bf16hi(u.z);
        v[8 * q + 6] = ptx::bf16lo(u.w); v[8 * q + 7] = ptx::bf16hi(u.w);
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float x = 0.f;
    if (j < n)
      x = fp32 ? static_cast<const float*>(rowp)[c0 + j]
               : __bfloat162float(static_cast<const __nv_bfloat16*>(rowp)[c0 + j]);
    v[j] = x;
  }
}

__device__ __forceinline__ void gstore32(void* rowp, int c0, int n, bool fp32, bool vec,
                                         const float (&v)[32]) {
  if (n >= 32 && vec) {
    if (fp32) {
      float4* p = reinterpret_cast<float4*>(static_cast<float*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q) p[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
      uint4* p = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        p[q] = make_uint4(ptx::pack_bf16x2(v[8 * q + 0], v[8 * q + 1]),
                          ptx::pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                          ptx::pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                          ptx::pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < n) {
      if (fp32) static_cast<float*>(rowp)[c0 + j] = v[j];
      else static_cast<__nv_bfloat16*>(rowp)[c0 + j] = __float2bfloat16_rn(v[j]);
    }
  }
}

// one element of a bf16 or fp32 matrix, as fp32 (and back, rounded to nearest)
__device__ __forceinline__ float ld_val(const void* base, int64_t idx, bool fp32) {
  return fp32 ? static_cast<const float*>(base)[idx]
              : __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}
__device__ __forceinline__ void st_val(void* base, int64_t idx, bool fp32, float v) {
  if (fp32) static_cast<float*>(base)[idx] = v;
  else static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}

__device__ __forceinline__ char* gptr(const void* base, int64_t ld, int64_t row, int64_t col,
                                      bool fp32) {
  return const_cast<char*>(static_cast<const char*>(base)) + (row * ld + col) * (fp32 ? 4 : 2);
}

// ------------------------------------------------------------------ bounded waits
// Waits for the phase of `bar` with the given parity. Gives up once the CTA
// has aborted or after limit_ns (then records the time-out and aborts the CTA).
// After an abort every wait returns at once, so all roles run to the end.
// try_wait with a suspend-time hint: the waiting thread sleeps until the phase
// completes or about 20 us pass, instead of spinning on the issue slots that
// the epilogue warps of its scheduler need.
__device__ __forceinline__ bool try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void wait_bar(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                         volatile int* abort_flag, int* err) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  while (!try_wait_sleep(bar, parity)) {
    if (*abort_flag) return;
    if (ptx::globaltimer() - t0 > limit_ns) {
      *abort_flag = 1;
      atomicCAS(err, 0, DEV_ERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void tensormap_acquire(const void* map) {
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

}  // namespace tile
}  // namespace himuon
