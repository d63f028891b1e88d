// Auxiliary kernels of libhimuon: per-matrix Frobenius norms (for the
// whole-matrix normalisation mode) and the self-test of the bounded wait.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace himuon {
namespace {

__device__ __forceinline__ float ld_elem(const void* base, int64_t idx, bool fp32) {
  return fp32 ? static_cast<const float*>(base)[idx]
              : __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}

// Part p covers NORM_ROWS_PER_PART rows of one matrix; its sum of squares of X
// (G, or for a step U = G + mu (mu M + G) / mu M + G) goes to partials[p].
__global__ void norm_partials(const MatDesc* __restrict__ descs, int ndesc,
                              const int64_t* __restrict__ part_start, float* __restrict__ partials,
                              StepArgs st) {
  const int64_t p = blockIdx.x;
  int lo = 0, hi = ndesc - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (part_start[mid] <= p) lo = mid; else hi = mid - 1;
  }
  const MatDesc& d = descs[lo];
  const int r0 = static_cast<int>(p - part_start[lo]) * NORM_ROWS_PER_PART;
  const int r1 = min(d.H, r0 + NORM_ROWS_PER_PART);
  const bool in32 = d.flags & F_IN_FP32;
  const bool m32 = !(d.flags & F_M_BF16);
  float acc = 0.f;
  for (int r = r0; r < r1; ++r) {
    for (int c = threadIdx.x; c < d.W; c += blockDim.x) {
      float v = ld_elem(d.in, static_cast<int64_t>(r) * d.ld_in + c, in32);
      if (st.enabled) {
        const float mn = fmaf(st.mu, ld_elem(d.mom, static_cast<int64_t>(r) * d.ld_mom + c, m32), v);
        v = st.nesterov ? fmaf(st.mu, mn, v) : mn;
      }
      acc = fmaf(v, v, acc);
    }
  }
  __shared__ float red[32];
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
    partials[p] = t;
  }
}

// One thread per matrix: sums its partials in order, stores 1 / (norm + eps).
__global__ void norm_finish(MatDesc* __restrict__ descs, int ndesc,
                            const int64_t* __restrict__ part_start,
                            const float* __restrict__ partials, float eps) {
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= ndesc) return;
  double t = 0.0;
  for (int64_t p = part_start[m]; p < part_start[m + 1]; ++p) t += partials[p];
  descs[m].norm_scale = static_cast<float>(1.0 / (sqrt(t) + static_cast<double>(eps)));
}

__global__ void wait_selftest_kernel(uint64_t wait_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
    // Nothing ever arrives on this barrier: the wait must give up by itself.
    if (!ptx::mbar_wait_bounded(b, 0, wait_ns)) atomicCAS(err, 0, DEV_ERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_matrix_norms(MatDesc* descs, int ndesc, const int64_t* part_start,
                                int64_t nparts_total, float* partials, float eps,
                                const StepArgs& st, cudaStream_t stream) {
  if (nparts_total <= 0) return cudaSuccess;
  norm_partials<<<static_cast<unsigned>(nparts_total), 256, 0, stream>>>(descs, ndesc, part_start,
                                                                          partials, st);
  norm_finish<<<(ndesc + 127) / 128, 128, 0, stream>>>(descs, ndesc, part_start, partials, eps);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t wait_ns, int* err, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(wait_ns, err);
  return cudaGetLastError();
}

}  // namespace himuon
