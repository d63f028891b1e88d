// Tiled Newton-Schulz for tiles of at most 32 x 32: one warp per tile, the whole
// tile in registers, products on the warp-level tensor-core instruction
// mma.sync.m16n8k16 (bf16 operands, fp32 accumulation).
//
// Method ("Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
// Optimization", abstract, sentences 3-5): every T x T tile X of a
// momentum-gradient matrix is normalised and iterated K times with
//   A = X X^T,  B = b A + c A^2,  X <- a X + B X,
// independently of every other tile.
//
// Why not tcgen05 here: a 32 x 32 tile is below the smallest tcgen05 product
// (M = 64), so the on-chip tcgen05 kernel stacks four of them into one 128-row
// operand and runs a 3K-long chain of dependent products and epilogues for just
// four tiles. Its products are tiny (32 x 32 x 32), the workload is bound by HBM
// (the pages' T = 32 map has about 240 flops per input byte at K = 5), and what
// limits it is latency, not tensor throughput. Here each warp owns one tile and
// a product is 16 mma.sync: the fp32 accumulator fragments of one product are,
// pair by pair, the bf16 A-operand fragments of the next, so a tile stays in its
// warp's registers for all K steps and 16 tiles per SM are in flight.
//
// Same arithmetic and rounding placement as the tcgen05 kernels: with
// e = a - min(a, 1.5) and C = B + e I,
//   X' = C X_bf + (a X - e X_bf)      (X in fp32, X_bf = bf16(X)),
// the input itself is the first step's operand (U_bf = bf16(U); the factor s
// enters as s^2 in A and s in X_1, so s U is never rounded), and
//   A_bf = bf16(s^2 U_bf U_bf^T)  (s^2 on the first step only),
//   C_bf = bf16(c A_bf A_bf + b A_bf + e I).
//
// Register layout (m16n8k16 fragments, g = lane / 4, t = lane % 4): a 32 x 32
// fp32 matrix is F[bm][bn][i], bm in {0, 1} (16-row blocks), bn in {0..3}
// (8-column blocks), element (16 bm + g + 8 (i >> 1), 8 bn + 2 t + (i & 1)).
// The bf16 A operand of the 16 x 16 block (bm, kb) is the four pairs
// F[bm][2kb][0,1], F[bm][2kb][2,3], F[bm][2kb+1][0,1], F[bm][2kb+1][2,3].
// For X X^T and A_bf A_bf (B[k][n] = M[n][k], M = X_bf or the symmetric A_bf)
// the B operand of (kb, bn) is two registers of M's A operand for row block
// bn / 2: no data movement. For C X_bf (B[k][n] = X_bf[k][n]) it is loaded
// transposed, with ldmatrix, from a per-warp shared copy of X_bf.
//
// Tiles are read and written row by row with the lanes along the columns
// (coalesced), through a per-warp fp32 shared tile that holds the processed
// matrix row-major; a wide tile (fewer rows than columns) is processed
// transposed (p(X)^T = p(X^T)), as on the other paths; a tile smaller than
// 32 x 32 (ragged edge, or T < 32) is zero-padded, which the map keeps zero.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace himuon {
namespace {

constexpr int MW = 8;                        // warps (tiles in flight) per block
constexpr int MTHREADS = MW * 32;
constexpr int US = 33;                       // fp32 tile row stride, words
constexpr int XS = 40;                       // bf16 tile row stride, elements (80 bytes:
                                             // conflict-free ldmatrix and pair stores)
constexpr uint32_t U_BYTES = 32 * US * 4;
constexpr uint32_t WARP_SMEM = U_BYTES + 32 * XS * 2;   // 6784 bytes, a multiple of 16

typedef float Frag[2][4][4];                 // fp32 32 x 32 in accumulator fragments
typedef uint32_t AFrag[2][2][4];             // bf16 32 x 32 in A-operand fragments

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four 8 x 8 bf16 matrices, transposed on the way: lane l gives the address of
// row l % 8 of matrix l / 8 and receives, from each matrix, the elements at rows
// 2 (l % 4), 2 (l % 4) + 1 of column l / 4 (the B-operand pattern).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void pack_a(const Frag& F, AFrag& A) {
#pragma unroll
  for (int bm = 0; bm < 2; ++bm)
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      A[bm][kb][0] = ptx::pack_bf16x2(F[bm][2 * kb][0], F[bm][2 * kb][1]);
      A[bm][kb][1] = ptx::pack_bf16x2(F[bm][2 * kb][2], F[bm][2 * kb][3]);
      A[bm][kb][2] = ptx::pack_bf16x2(F[bm][2 * kb + 1][0], F[bm][2 * kb + 1][1]);
      A[bm][kb][3] = ptx::pack_bf16x2(F[bm][2 * kb + 1][2], F[bm][2 * kb + 1][3]);
    }
}

// Packed fp32 pairs (one instruction for two adjacent columns, the same
// roundings as two scalar operations).
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
// the two bf16 values of an A-operand register, as a packed fp32 pair
__device__ __forceinline__ uint64_t a_pair(uint32_t r) { return pk2(ptx::bf16lo(r), ptx::bf16hi(r)); }
// F *= x for the whole fragment set
__device__ __forceinline__ void scale_frag(Frag& F, float x) {
  const uint64_t x2 = pk2(x, x);
#pragma unroll
  for (int bm = 0; bm < 2; ++bm)
#pragma unroll
    for (int bn = 0; bn < 4; ++bn)
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const uint64_t v = mul2(pk2(F[bm][bn][i], F[bm][bn][i + 1]), x2);
        upk2(v, F[bm][bn][i], F[bm][bn][i + 1]);
      }
}

// D = M M^T from M's own A-operand fragments (the B operand of (kb, bn) is row
// block bn / 2 of M: registers (bn & 1) and 2 + (bn & 1) of its k-block kb).
__device__ __forceinline__ void gram(const AFrag& M, Frag& D) {
#pragma unroll
  for (int bm = 0; bm < 2; ++bm)
#pragma unroll
    for (int bn = 0; bn < 4; ++bn) {
#pragma unroll
      for (int i = 0; i < 4; ++i) D[bm][bn][i] = 0.f;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
        mma16816(D[bm][bn], M[bm][kb], M[bn >> 1][kb][bn & 1], M[bn >> 1][kb][2 + (bn & 1)]);
    }
}

template <bool STEP>
__global__ void __launch_bounds__(MTHREADS, 2)
    ns_mma32_kernel(const MatDesc* __restrict__ descs, int ndesc, int64_t tile_begin,
                    int64_t tile_end, NSArgs ns, StepArgs st) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  float* su = reinterpret_cast<float*>(smem + warp * WARP_SMEM);
  __nv_bfloat16* sx = reinterpret_cast<__nv_bfloat16*>(smem + warp * WARP_SMEM + U_BYTES);
  const uint32_t sx_addr = ptx::smem_u32(sx);
  const int T = ns.T, K = ns.K;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * MW;

  for (int64_t tile = tile_begin + static_cast<int64_t>(blockIdx.x) * MW + warp; tile < tile_end;
       tile += nwarps) {
    const int mi = find_matrix(descs, ndesc, tile);
    const MatDesc& d = descs[mi];
    const int64_t lt = tile - d.tile_start;
    const int i0 = static_cast<int>(lt / d.tiles_w) * T, j0 = static_cast<int>(lt % d.tiles_w) * T;
    const int h = min(T, d.H - i0), w = min(T, d.W - j0);
    const bool tr = h < w;
    const bool in32 = d.flags & F_IN_FP32, m16 = d.flags & F_M_BF16, out32 = d.flags & F_OUT_FP32;

    // the rows of this warp's next tile (G, and M for a step) into L2 while
    // this one is processed: lane l takes row l (one 32-element row segment
    // starts at a multiple of T elements, so it spans at most two lines)
    if (tile + nwarps < tile_end) {
      const int64_t nt = tile + nwarps;
      const MatDesc& dn = descs[find_matrix(descs, ndesc, nt)];
      const int64_t nlt = nt - dn.tile_start;
      const int ni0 = static_cast<int>(nlt / dn.tiles_w) * T, nj0 = static_cast<int>(nlt % dn.tiles_w) * T;
      if (lane < min(T, dn.H - ni0)) {
        const int es = (dn.flags & F_IN_FP32) ? 4 : 2;
        const char* gp = static_cast<const char*>(dn.in) + ((ni0 + lane) * dn.ld_in + nj0) * es;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(gp));
        if (STEP) {
          const int ms = (dn.flags & F_M_BF16) ? 2 : 4;
          const char* mp = static_cast<const char*>(dn.mom) + ((ni0 + lane) * dn.ld_mom + nj0) * ms;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(mp));
        }
      }
    }

    // ---- U = G (or, for a step, the Nesterov/plain momentum direction, with
    // M <- mu M + G written back), row by row, into the shared tile at its
    // processed position; zeros outside the tile.
    float ssq = 0.f;
    {
      // one predicated read-only load per row, all issued before any is used;
      // the dtype is chosen once per tile, outside the row loop
      float u[32];
      const bool col_ok = lane < w;
      const int hv = col_ok ? h : 0;           // rows this lane loads
      if (in32) {
        const float* gp = static_cast<const float*>(d.in) + static_cast<int64_t>(i0) * d.ld_in + j0 + lane;
#pragma unroll
        for (int i = 0; i < 32; ++i) u[i] = (i < hv) ? __ldg(gp + static_cast<int64_t>(i) * d.ld_in) : 0.f;
      } else {
        const __nv_bfloat16* gp =
            static_cast<const __nv_bfloat16*>(d.in) + static_cast<int64_t>(i0) * d.ld_in + j0 + lane;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          u[i] = (i < hv) ? __bfloat162float(__ldg(gp + static_cast<int64_t>(i) * d.ld_in)) : 0.f;
      }
      if (STEP) {
        float m[32];
        if (m16) {
          const __nv_bfloat16* mp =
              static_cast<const __nv_bfloat16*>(d.mom) + static_cast<int64_t>(i0) * d.ld_mom + j0 + lane;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            m[i] = (i < hv) ? __bfloat162float(mp[static_cast<int64_t>(i) * d.ld_mom]) : 0.f;
        } else {
          const float* mp = static_cast<const float*>(d.mom) + static_cast<int64_t>(i0) * d.ld_mom + j0 + lane;
#pragma unroll
          for (int i = 0; i < 32; ++i) m[i] = (i < hv) ? mp[static_cast<int64_t>(i) * d.ld_mom] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (i < hv) {
            const float mn = fmaf(st.mu, m[i], u[i]);
            const int64_t mo = static_cast<int64_t>(i0 + i) * d.ld_mom + j0 + lane;
            if (m16) static_cast<__nv_bfloat16*>(d.mom)[mo] = __float2bfloat16_rn(mn);
            else static_cast<float*>(d.mom)[mo] = mn;
            u[i] = st.nesterov ? fmaf(st.mu, mn, u[i]) : mn;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        ssq = fmaf(u[i], u[i], ssq);
        su[tr ? lane * US + i : i * US + lane] = u[i];
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
    float s = 1.f;
    if (ns.norm == NORM_TILE) s = 1.f / (sqrtf(ssq) + ns.eps);
    else if (ns.norm == NORM_MATRIX) s = d.norm_scale;
    __syncwarp();

    float scale_out = s;                      // K = 0: the output is s U
    if (K > 0) {
      // ---- X = U (unnormalised) in fragments; R = a X - e X_bf
      Frag R;
      AFrag XA;
#pragma unroll
      for (int bm = 0; bm < 2; ++bm)
#pragma unroll
        for (int bn = 0; bn < 4; ++bn)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            R[bm][bn][i] = su[(16 * bm + g + 8 * (i >> 1)) * US + 8 * bn + 2 * t + (i & 1)];
      scale_out = 1.f;
#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        const StepCoef cf = step_coef(ns, k);  // this step's (a, b, c) and shift e
        const float e = cf.e;
        const bool has_c = cf.has_c;
        // this lane's diagonal positions: F[bm][2bm][0 | 1] and F[bm][2bm+1][2 | 3]
        const float ed0 = (g == 2 * t) ? e : 0.f, ed1 = (g == 2 * t + 1) ? e : 0.f;
        // R holds X here: its bf16 operand, and R = a X - e X_bf
        pack_a(R, XA);
#pragma unroll
        for (int bm = 0; bm < 2; ++bm)
#pragma unroll
          for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int row = 16 * bm + g + 8 * (q & 1), col = 16 * kb + 2 * t + 8 * (q >> 1);
              *reinterpret_cast<uint32_t*>(sx + row * XS + col) = XA[bm][kb][q];
            }
        {
          const uint64_t a2 = pk2(cf.a, cf.a), ne2 = pk2(-e, -e);
#pragma unroll
          for (int bm = 0; bm < 2; ++bm)
#pragma unroll
            for (int bn = 0; bn < 4; ++bn)
#pragma unroll
              for (int i = 0; i < 4; i += 2) {
                const uint64_t xb = a_pair(XA[bm][bn >> 1][2 * (bn & 1) + (i >> 1)]);
                const uint64_t v = fma2(a2, pk2(R[bm][bn][i], R[bm][bn][i + 1]), mul2(ne2, xb));
                upk2(v, R[bm][bn][i], R[bm][bn][i + 1]);
              }
        }

        // ---- A = X_bf X_bf^T  ->  A_bf = bf16(s^2 A)  (or C directly when c = 0)
        Frag D;
        gram(XA, D);
        const float s2 = (k == 0) ? s * s : 1.f;
        AFrag AB;
        if (has_c) {
          if (k == 0) scale_frag(D, s2);
          pack_a(D, AB);
          // ---- R_A = A_bf A_bf  ->  C = c A_bf A_bf + b A_bf + e I
          gram(AB, D);
          const uint64_t c2 = pk2(cf.c, cf.c), b2 = pk2(cf.b, cf.b);
#pragma unroll
          for (int bm = 0; bm < 2; ++bm)
#pragma unroll
            for (int bn = 0; bn < 4; ++bn)
#pragma unroll
              for (int i = 0; i < 4; i += 2) {
                const uint64_t ab = a_pair(AB[bm][bn >> 1][2 * (bn & 1) + (i >> 1)]);
                const uint64_t v = fma2(c2, pk2(D[bm][bn][i], D[bm][bn][i + 1]), mul2(b2, ab));
                upk2(v, D[bm][bn][i], D[bm][bn][i + 1]);
              }
        } else {
          scale_frag(D, cf.b * s2);
        }
#pragma unroll
        for (int bm = 0; bm < 2; ++bm) {
          D[bm][2 * bm][0] += ed0;
          D[bm][2 * bm][1] += ed1;
          D[bm][2 * bm + 1][2] += ed0;
          D[bm][2 * bm + 1][3] += ed1;
        }
        pack_a(D, AB);                        // C_bf

        // ---- X' = C X_bf + (a X - e X_bf): B operand X_bf from the shared copy
        __syncwarp();
#pragma unroll
        for (int bn = 0; bn < 4; ++bn) {
          uint32_t b00, b01, b10, b11;
          ldsm_x4_trans(sx_addr + static_cast<uint32_t>((lane * XS + 8 * bn) * 2), b00, b01, b10, b11);
#pragma unroll
          for (int bm = 0; bm < 2; ++bm) {
            mma16816(R[bm][bn], AB[bm][0], b00, b01);
            mma16816(R[bm][bn], AB[bm][1], b10, b11);
          }
        }
        if (k == 0) scale_frag(R, s);         // X_1 = s (C U_bf + a U - e U_bf)
        __syncwarp();                         // the shared X_bf is rewritten next step
      }
      // the result into the shared tile (processed coordinates)
#pragma unroll
      for (int bm = 0; bm < 2; ++bm)
#pragma unroll
        for (int bn = 0; bn < 4; ++bn)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            su[(16 * bm + g + 8 * (i >> 1)) * US + 8 * bn + 2 * t + (i & 1)] = R[bm][bn][i];
      __syncwarp();
    }

    // ---- write back row by row (lanes along the columns): the output, or the
    // weight update W <- wd W - lr s O
    if (lane < w) {
#pragma unroll 4
      for (int i = 0; i < h; ++i) {
        const float o = scale_out * su[tr ? lane * US + i : i * US + lane];
        char* p = static_cast<char*>(d.out) +
                  (static_cast<int64_t>(i0 + i) * d.ld_out + j0 + lane) * (out32 ? 4 : 2);
        float v = o;
        if (STEP) {
          const float wv = out32 ? *reinterpret_cast<const float*>(p)
                                 : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
          v = fmaf(-d.upd_scale, o, wv * st.wd_factor);
        }
        if (out32) *reinterpret_cast<float*>(p) = v;
        else *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
      }
    }
    __syncwarp();                             // the shared tile is refilled next
  }
}

template <bool STEP>
cudaError_t launch_m(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                     const NSArgs& ns, const StepArgs& st, int num_sms, cudaStream_t stream) {
  const uint32_t smem = MW * WARP_SMEM;
  cudaError_t e = cudaFuncSetAttribute(ns_mma32_kernel<STEP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t want = (tile_end - tile_begin + MW - 1) / MW;
  const int grid = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(num_sms) * 2));
  ns_mma32_kernel<STEP><<<grid, MTHREADS, smem, stream>>>(descs, ndesc, tile_begin, tile_end, ns, st);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_mma32(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                            const NSArgs& ns, const StepArgs& st, int num_sms, cudaStream_t stream) {
  if (tile_end <= tile_begin) return cudaSuccess;
  if (ns.T < 1 || ns.T > 32) return cudaErrorInvalidValue;
  return st.enabled ? launch_m<true>(descs, ndesc, tile_begin, tile_end, ns, st, num_sms, stream)
                    : launch_m<false>(descs, ndesc, tile_begin, tile_end, ns, st, num_sms, stream);
}

}  // namespace himuon
