// fp32 validation path of the tiled Newton-Schulz map (CUDA cores, fp32 FMA).
//
// Same map as the tensor-core path ("Hierarchical Muon: Tiled Newton-Schulz
// Updates for Efficient Muon Optimization", abstract, sentences 3-5), kept in
// fp32 end to end so that it can be held to a tight tolerance against the fp64
// oracle. Tiles are zero-padded to P x P in a scratch buffer (zero rows and
// columns stay zero through the polynomial and do not change the Frobenius
// norm, so the valid block is unaffected), and every NS step runs as three
// batched SIMT GEMMs over all tiles of a sub-batch:
//   A = X X^T;  B = c A A + b A;  X' = B X + a X.
// Any tile size works, including one tile covering the whole matrix.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace himuon {
namespace {

__device__ __forceinline__ float ld_elem(const void* base, int64_t idx, bool fp32) {
  return fp32 ? static_cast<const float*>(base)[idx]
              : __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
}
__device__ __forceinline__ void st_elem(void* base, int64_t idx, bool fp32, float v) {
  if (fp32) static_cast<float*>(base)[idx] = v;
  else static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
}

struct TileLoc {
  const MatDesc* d;
  int i0, j0, h, w;
};

__device__ __forceinline__ TileLoc locate(const MatDesc* descs, int ndesc, int64_t tile, int T) {
  const int mi = find_matrix(descs, ndesc, tile);
  const MatDesc* d = &descs[mi];
  const int64_t lt = tile - d->tile_start;
  TileLoc L;
  L.d = d;
  L.i0 = static_cast<int>(lt / d->tiles_w) * T;
  L.j0 = static_cast<int>(lt % d->tiles_w) * T;
  L.h = min(T, d->H - L.i0);
  L.w = min(T, d->W - L.j0);
  return L;
}

// One CTA per tile: copy the tile into X (P x P, zero padded). For a step,
// apply the momentum update first (M written back) and gather U.
__global__ void f32_gather(const MatDesc* __restrict__ descs, int ndesc, int64_t tile0, int T,
                           int P, float* __restrict__ X, StepArgs st) {
  const TileLoc L = locate(descs, ndesc, tile0 + blockIdx.x, T);
  const MatDesc& d = *L.d;
  float* x = X + static_cast<int64_t>(blockIdx.x) * P * P;
  const bool in32 = d.flags & F_IN_FP32;
  const bool m32 = !(d.flags & F_M_BF16);
  for (int64_t e = threadIdx.x; e < static_cast<int64_t>(P) * P; e += blockDim.x) {
    const int r = static_cast<int>(e / P), c = static_cast<int>(e % P);
    float v = 0.f;
    if (r < L.h && c < L.w) {
      const int64_t gi = static_cast<int64_t>(L.i0 + r) * d.ld_in + (L.j0 + c);
      v = ld_elem(d.in, gi, in32);
      if (st.enabled) {
        const int64_t mi = static_cast<int64_t>(L.i0 + r) * d.ld_mom + (L.j0 + c);
        const float mn = fmaf(st.mu, ld_elem(d.mom, mi, m32), v);
        st_elem(d.mom, mi, m32, mn);
        v = st.nesterov ? fmaf(st.mu, mn, v) : mn;
      }
    }
    x[e] = v;
  }
}

// One CTA per tile: scale by 1 / (||X||_F + eps) (tile mode) or by the
// matrix's precomputed factor (matrix mode).
__global__ void f32_normalise(const MatDesc* __restrict__ descs, int ndesc, int64_t tile0, int T,
                             int P, float* __restrict__ X, int norm, float eps) {
  const TileLoc L = locate(descs, ndesc, tile0 + blockIdx.x, T);
  float* x = X + static_cast<int64_t>(blockIdx.x) * P * P;
  const int64_t n = static_cast<int64_t>(P) * P;
  __shared__ float red[32];
  float s;
  if (norm == NORM_TILE) {
    float acc = 0.f;
    for (int64_t e = threadIdx.x; e < n; e += blockDim.x) acc = fmaf(x[e], x[e], acc);
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) t += red[i];
      red[0] = 1.f / (sqrtf(t) + eps);
    }
    __syncthreads();
    s = red[0];
  } else {
    s = L.d->norm_scale;
  }
  for (int64_t e = threadIdx.x; e < n; e += blockDim.x) x[e] *= s;
}

// Batched D = alpha * A op(B) + beta * C over P x P matrices (batch = blockIdx.z).
// op(B) = B^T when NT. 64 x 64 output block per CTA, 4 x 4 per thread.
template <bool NT>
__global__ void __launch_bounds__(256) f32_gemm(const float* __restrict__ A,
                                                const float* __restrict__ B,
                                                const float* __restrict__ C, float* __restrict__ D,
                                                int P, float alpha, float beta) {
  const int64_t off = static_cast<int64_t>(blockIdx.z) * P * P;
  A += off;
  B += off;
  D += off;
  if (C) C += off;
  __shared__ float As[16][68];
  __shared__ float Bs[16][68];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < P; k0 += 16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = threadIdx.x + i * 256;
      const int mm = e >> 4, kk = e & 15;
      const int gm = m0 + mm, gk = k0 + kk;
      As[kk][mm] = (gm < P && gk < P) ? A[static_cast<int64_t>(gm) * P + gk] : 0.f;
      if (NT) {
        const int gn = n0 + mm;
        Bs[kk][mm] = (gn < P && gk < P) ? B[static_cast<int64_t>(gn) * P + gk] : 0.f;
      } else {
        const int kb = e >> 6, nb = e & 63;
        const int gkb = k0 + kb, gn = n0 + nb;
        Bs[kb][nb] = (gkb < P && gn < P) ? B[static_cast<int64_t>(gkb) * P + gn] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty + 16 * i;
    if (gm >= P) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx + 16 * j;
      if (gn >= P) continue;
      const int64_t idx = static_cast<int64_t>(gm) * P + gn;
      float v = alpha * acc[i][j];
      if (C) v = fmaf(beta, C[idx], v);
      D[idx] = v;
    }
  }
}

// One CTA per tile: write the valid block to the output, or apply the update
// W <- wd_factor * W - upd_scale * X for a step.
__global__ void f32_scatter(const MatDesc* __restrict__ descs, int ndesc, int64_t tile0, int T,
                            int P, const float* __restrict__ X, StepArgs st) {
  const TileLoc L = locate(descs, ndesc, tile0 + blockIdx.x, T);
  const MatDesc& d = *L.d;
  const float* x = X + static_cast<int64_t>(blockIdx.x) * P * P;
  const bool out32 = d.flags & F_OUT_FP32;
  for (int64_t e = threadIdx.x; e < static_cast<int64_t>(L.h) * L.w; e += blockDim.x) {
    const int r = static_cast<int>(e / L.w), c = static_cast<int>(e % L.w);
    const int64_t oi = static_cast<int64_t>(L.i0 + r) * d.ld_out + (L.j0 + c);
    const float v = x[static_cast<int64_t>(r) * P + c];
    if (st.enabled) {
      const float wv = ld_elem(d.out, oi, out32);
      st_elem(d.out, oi, out32, fmaf(-d.upd_scale, v, wv * st.wd_factor));
    } else {
      st_elem(d.out, oi, out32, v);
    }
  }
}

}  // namespace

cudaError_t launch_ns_fp32(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                           int T, int P, const NSArgs& ns, const StepArgs& st, float* scratch,
                           int64_t nb, cudaStream_t stream) {
  const int64_t pp = static_cast<int64_t>(P) * P;
  for (int64_t t0 = tile_begin; t0 < tile_end; t0 += nb) {
    const int n = static_cast<int>(std::min<int64_t>(nb, tile_end - t0));
    float* X = scratch;
    float* A = scratch + static_cast<int64_t>(n) * pp;
    float* B = scratch + 2 * static_cast<int64_t>(n) * pp;
    f32_gather<<<n, 256, 0, stream>>>(descs, ndesc, t0, T, P, X, st);
    if (ns.norm != NORM_NONE) f32_normalise<<<n, 256, 0, stream>>>(descs, ndesc, t0, T, P, X, ns.norm, ns.eps);
    const dim3 g((P + 63) / 64, (P + 63) / 64, n);
    for (int k = 0; k < ns.K; ++k) {
      f32_gemm<true><<<g, 256, 0, stream>>>(X, X, nullptr, A, P, 1.f, 0.f);
      const StepCoef cf = step_coef(ns, k);
      f32_gemm<false><<<g, 256, 0, stream>>>(A, A, A, B, P, cf.c, cf.b);
      f32_gemm<false><<<g, 256, 0, stream>>>(B, X, X, A, P, 1.f, cf.a);
      std::swap(X, A);
    }
    f32_scatter<<<n, 256, 0, stream>>>(descs, ndesc, t0, T, P, X, st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace himuon
