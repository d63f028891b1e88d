// Tiled Newton-Schulz on tcgen05 tensor cores, T = 128, tile resident on chip.
//
// Method ("Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
// Optimization", abstract, sentences 3-5): every T x T tile X of a
// momentum-gradient matrix is normalised and then iterated K times with
//   A = X X^T,  B = b A + c A^2,  X <- a X + B X,
// independently of all other tiles. The three products per step are dense
// 128 x 128 x 128 contractions, issued here as tcgen05.mma (bf16 operands, fp32
// accumulation in tensor memory).
//
// One CTA of 128 threads owns one tile at a time; thread r owns tile row r,
// which is also TMEM lane r of every accumulator. Two CTAs share an SM (shared
// memory is padded to enforce it) so that one CTA's epilogue overlaps the
// other's MMAs. The CTA is persistent and walks the flat tile list of a launch,
// which may span many matrices (cross-layer batching).
//
// On-chip state of a tile:
//   sX  (smem, 32 KB)  X in bf16: MMA operand of X X^T (K-major) and of B X
//                      (MN-major); 128-byte swizzled, two 64-column halves.
//   sA  (smem, 32 KB)  A in bf16 (operand of A A), then B in bf16 (operand of B X).
//   TMEM cols [0,128)  fp32 accumulator: A, then A^2, then B X.
//   TMEM cols [128,256) X in fp32, used for the a X term, so that the iterate is
//                      rounded to bf16 only where it feeds a product.
// Normalisation: on the first step the scale s = 1 / (||X||_F + eps) is folded
// into the epilogues (||X||_F^2 = trace(X X^T) read from the first accumulator),
// so the unnormalised bf16 input is used as the operand without a rounding.
//
// Loading: 16-byte (or scalar, for unaligned rows) global loads by the owning
// thread. For a HiMuon step the loader also applies momentum (M <- mu M + G,
// U = G + mu M) and the final epilogue applies the weight update in place, so
// neither U nor the NS output ever goes to HBM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace himuon {
namespace {

constexpr int TT = 128;                 // tile size
constexpr int NTHR = 128;               // threads per CTA (one per tile row)
constexpr uint32_t SMEM_X = 0;
constexpr uint32_t SMEM_A = 32768;
constexpr uint32_t SMEM_BAR = 65536;
// 96 KB + alignment slack: more than a third of the SM's shared memory, so at
// most two CTAs are resident per SM and their TMEM (2 x 256 columns) always fits.
constexpr uint32_t SMEM_BYTES = 96 * 1024 + 1024;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t XF_COL = 128;

// Byte offset of 16-byte chunk `c16` (0..15, i.e. columns 8*c16..8*c16+7) of row
// `r` in a 128 x 128 bf16 tile stored as two 64-column halves of 128 rows x
// 128 bytes with the 128-byte swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t sw128(int r, int c16) {
  return static_cast<uint32_t>((c16 >> 3) * 16384 + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}

// Writes 32 fp32 values (columns 32*ch .. 32*ch+31 of row r) as bf16 into a tile.
__device__ __forceinline__ void put_bf16_row32(uint32_t tile, int r, int ch, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    ptx::st_shared_v4(tile + sw128(r, ch * 4 + q), ptx::pack_bf16x2(v[8 * q + 0], v[8 * q + 1]),
                      ptx::pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                      ptx::pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                      ptx::pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  }
}

__device__ __forceinline__ void get_bf16_row32(uint32_t tile, int r, int ch, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u = ptx::ld_shared_v4(tile + sw128(r, ch * 4 + q));
    v[8 * q + 0] = ptx::bf16lo(u.x); v[8 * q + 1] = ptx::bf16hi(u.x);
    v[8 * q + 2] = ptx::bf16lo(u.y); v[8 * q + 3] = ptx::bf16hi(u.y);
    v[8 * q + 4] = ptx::bf16lo(u.z); v[8 * q + 5] = ptx::bf16hi(u.z);
    v[8 * q + 6] = ptx::bf16lo(u.w); v[8 * q + 7] = ptx::bf16hi(u.w);
  }
}

// ---- global row segment access: 32 elements starting at column c0 of a row,
// `n` of them valid (0..32). Vector path when all 32 are valid and `vec`.
__device__ __forceinline__ void load_seg(const void* rowp, int c0, int n, bool fp32, bool vec,
                                         float (&v)[32]) {
  if (n >= 32 && vec) {
    if (fp32) {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 f = p[q];
        v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
      }
    } else {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 u = p[q];
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
    if (j < n) {
      x = fp32 ? static_cast<const float*>(rowp)[c0 + j]
               : __bfloat162float(static_cast<const __nv_bfloat16*>(rowp)[c0 + j]);
    }
    v[j] = x;
  }
}

__device__ __forceinline__ void store_seg(void* rowp, int c0, int n, bool fp32, bool vec,
                                          const float (&v)[32]) {
  if (n >= 32 && vec) {
    if (fp32) {
      float4* p = reinterpret_cast<float4*>(static_cast<float*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q) p[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
      uint4* p = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(rowp) + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p[q] = make_uint4(ptx::pack_bf16x2(v[8 * q + 0], v[8 * q + 1]),
                          ptx::pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                          ptx::pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                          ptx::pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
      }
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

__device__ __forceinline__ const char* row_ptr(const void* base, int64_t ld, int row, int col,
                                               bool fp32) {
  const int64_t esz = fp32 ? 4 : 2;
  return static_cast<const char*>(base) + (static_cast<int64_t>(row) * ld + col) * esz;
}

template <bool STEP>
__global__ void __launch_bounds__(NTHR, 1)
    ns_tc128_kernel(const MatDesc* __restrict__ descs, int ndesc, int64_t tile_begin,
                    int64_t tile_end, NSArgs ns, StepArgs st, uint64_t wait_ns,
                    int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ float red[4];
  __shared__ int abort_flag;

  const uint32_t sbase = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sX = sbase + SMEM_X;
  const uint32_t sA = sbase + SMEM_A;
  const uint32_t bar = sbase + SMEM_BAR;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int r = tid;

  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  const uint32_t tbase = tmem_slot;
  const uint32_t t_acc = tbase + ACC_COL;                         // MMA destination
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t t_acc_w = tbase + lane_off + ACC_COL;            // this warp's lanes
  const uint32_t t_xf_w = tbase + lane_off + XF_COL;

  constexpr uint32_t IDESC_KK = ptx::idesc_bf16_f32(128, 128, false, false);
  constexpr uint32_t IDESC_KM = ptx::idesc_bf16_f32(128, 128, false, true);

  uint32_t phase = 0;
  const int K = ns.K;
  // Part (a - d) of the a X term is moved into the bf16 operand C = B + (a - d) I,
  // d = min(a, 1.5): the spectrum of B (about [-2.8, 0] for the quintic) is
  // then centred on zero, which shrinks the bf16 rounding of C relative to the
  // result a + B where a + b s^2 + c s^4 nearly cancels (rank-1 tiles).
  const float shift = ns.a > 1.5f ? ns.a - 1.5f : 0.f;

  // Waits for the MMAs committed last; one thread polls (bounded), all sync.
  auto wait_mma = [&]() -> bool {
    if (tid == 0) {
      if (!ptx::mbar_wait_bounded(bar, phase, wait_ns)) {
        abort_flag = 1;
        atomicCAS(err, 0, DEV_ERR_TIMEOUT);
      }
    }
    phase ^= 1u;
    __syncthreads();
    ptx::tc_fence_after();
    return abort_flag == 0;
  };

  // Issues the 8 K-slices of one 128 x 128 x 128 product and commits them.
  // a_base/b_base: smem tiles; b_mn: B operand read MN-major (rows of X as K).
  auto issue = [&](uint32_t a_base, uint32_t b_base, bool b_mn) {
    if (tid == 0) {
      ptx::tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a_addr = a_base + (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint64_t ad = ptx::sdesc_sw128(a_addr, 16, 1024);
        uint64_t bd;
        if (b_mn) {
          // K rows kk*16 .. kk*16+15 of X; 64-column halves 16 KB apart (LBO),
          // 8-row groups 1 KB apart (SBO).
          bd = ptx::sdesc_sw128(b_base + kk * 2048, 16384, 1024);
        } else {
          bd = ptx::sdesc_sw128(b_base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        }
        ptx::umma_bf16(t_acc, ad, bd, b_mn ? IDESC_KM : IDESC_KK, kk > 0 ? 1u : 0u);
      }
      ptx::umma_commit(bar);
    }
  };

  auto sync_for_mma = [&]() {
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
  };

  for (int64_t tile = tile_begin + blockIdx.x; tile < tile_end; tile += gridDim.x) {
    const int mi = find_matrix(descs, ndesc, tile);
    const MatDesc& d = descs[mi];
    const int64_t lt = tile - d.tile_start;
    const int ti = static_cast<int>(lt / d.tiles_w);
    const int tj = static_cast<int>(lt % d.tiles_w);
    const int i0 = ti * TT, j0 = tj * TT;
    const int h = min(TT, d.H - i0);
    const int w = min(TT, d.W - j0);
    const int flags = d.flags;
    const bool in32 = flags & F_IN_FP32, out32 = flags & F_OUT_FP32;
    const bool row_ok = r < h;

    // ---------------- load (and momentum): X -> TMEM xf (fp32) and sX (bf16)
    {
      const char* gp = row_ok ? row_ptr(d.in, d.ld_in, i0 + r, j0, in32) : nullptr;
      char* mp = nullptr;
      const bool m16 = flags & F_M_BF16;
      if (STEP && row_ok) mp = const_cast<char*>(row_ptr(d.mom, d.ld_mom, i0 + r, j0, !m16));
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        const int n = row_ok ? max(0, min(32, w - ch * 32)) : 0;
        float v[32];
        load_seg(gp, ch * 32, n, in32, flags & F_IN_VEC, v);
        if (STEP) {
          float m[32];
          load_seg(mp, ch * 32, n, !m16, flags & F_M_VEC, m);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float mn = fmaf(st.mu, m[j], v[j]);
            m[j] = mn;
            v[j] = st.nesterov ? fmaf(st.mu, mn, v[j]) : mn;
          }
          if (n > 0) store_seg(mp, ch * 32, n, !m16, flags & F_M_VEC, m);
        }
        ptx::tmem_st32(t_xf_w + ch * 32, v);
        put_bf16_row32(sX, r, ch, v);
      }
      ptx::tmem_wait_st();
    }
    sync_for_mma();

    // ---------------- normalisation factor
    float s = 1.f;
    if (ns.norm == NORM_MATRIX) s = d.norm_scale;

    if (K == 0) {
      if (ns.norm == NORM_TILE) {
        float acc = 0.f;
        for (int ch = 0; ch < 4; ++ch) {
          float xp[32];
          ptx::tmem_ld32_sync(t_xf_w + ch * 32, xp);
#pragma unroll
          for (int j = 0; j < 32; ++j) acc = fmaf(xp[j], xp[j], acc);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        s = 1.f / (sqrtf(((red[0] + red[1]) + red[2]) + red[3]) + ns.eps);
      }
      for (int ch = 0; ch < 4; ++ch) {
        float xp[32];
        ptx::tmem_ld32_sync(t_xf_w + ch * 32, xp);
#pragma unroll
        for (int j = 0; j < 32; ++j) xp[j] *= s;
        if (row_ok) {
          const int n = max(0, min(32, w - ch * 32));
          if (n > 0) {
            char* op = const_cast<char*>(row_ptr(d.out, d.ld_out, i0 + r, j0, out32));
            if (STEP) {
              float wv[32];
              load_seg(op, ch * 32, n, out32, flags & F_OUT_VEC, wv);
#pragma unroll
              for (int j = 0; j < 32; ++j) wv[j] = fmaf(-d.upd_scale, xp[j], wv[j] * st.wd_factor);
              store_seg(op, ch * 32, n, out32, flags & F_OUT_VEC, wv);
            } else {
              store_seg(op, ch * 32, n, out32, flags & F_OUT_VEC, xp);
            }
          }
        }
      }
      ptx::tc_fence_before();
      __syncthreads();
      continue;
    }

#pragma unroll 1
    for (int k = 0; k < K; ++k) {
      // ---- A = X X^T
      issue(sX, sX, false);
      if (!wait_mma()) goto teardown;
      if (k == 0 && ns.norm == NORM_TILE) {
        // ||X||_F^2 = trace(X X^T); warp w's rows have their diagonal in
        // accumulator columns 32w .. 32w+31.
        float v[32];
        ptx::tmem_ld32_sync(t_acc_w + warp * 32, v);
        float dg = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) dg = (j == lane) ? v[j] : dg;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dg += __shfl_xor_sync(0xffffffffu, dg, o);
        if (lane == 0) red[warp] = dg;
        __syncthreads();
        s = 1.f / (sqrtf(((red[0] + red[1]) + red[2]) + red[3]) + ns.eps);
      }
      {
        const float s2 = (k == 0) ? s * s : 1.f;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float v[32];
          ptx::tmem_ld32_sync(t_acc_w + ch * 32, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= s2;
          put_bf16_row32(sA, r, ch, v);
        }
      }
      sync_for_mma();

      // ---- A^2 = A A  (A symmetric: its rows serve as the K-major B operand)
      issue(sA, sA, false);
      if (!wait_mma()) goto teardown;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        float a2[32], av[32];
        get_bf16_row32(sA, r, ch, av);
        ptx::tmem_ld32_sync(t_acc_w + ch * 32, a2);
#pragma unroll
        for (int j = 0; j < 32; ++j) av[j] = fmaf(ns.c, a2[j], ns.b * av[j]);
        if (ch == warp) {                 // this row's diagonal element: + (a - d)
#pragma unroll
          for (int j = 0; j < 32; ++j) av[j] += (j == lane) ? shift : 0.f;
        }
        put_bf16_row32(sA, r, ch, av);   // C = b A + c A^2 + (a - d) I, in place of A
      }
      sync_for_mma();

      // ---- B X
      issue(sA, sX, true);
      if (!wait_mma()) goto teardown;
      {
        const float sb = (k == 0) ? s : 1.f;
        const bool last = (k + 1 == K);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          float bx[32], xp[32], xb[32];
          ptx::tmem_ld32x2_sync(t_acc_w + ch * 32, bx, t_xf_w + ch * 32, xp);
          get_bf16_row32(sX, r, ch, xb);
          // X' = C X_bf + a X - (a - d) X_bf  (= a X + B X_bf exactly)
#pragma unroll
          for (int j = 0; j < 32; ++j) xp[j] = sb * fmaf(-shift, xb[j], fmaf(ns.a, xp[j], bx[j]));
          if (!last) {
            ptx::tmem_st32(t_xf_w + ch * 32, xp);
            put_bf16_row32(sX, r, ch, xp);
          } else if (row_ok) {
            const int n = max(0, min(32, w - ch * 32));
            if (n > 0) {
              char* op = const_cast<char*>(row_ptr(d.out, d.ld_out, i0 + r, j0, out32));
              if (STEP) {
                float wv[32];
                load_seg(op, ch * 32, n, out32, flags & F_OUT_VEC, wv);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  wv[j] = fmaf(-d.upd_scale, xp[j], wv[j] * st.wd_factor);
                store_seg(op, ch * 32, n, out32, flags & F_OUT_VEC, wv);
              } else {
                store_seg(op, ch * 32, n, out32, flags & F_OUT_VEC, xp);
              }
            }
          }
        }
        ptx::tmem_wait_st();
      }
      sync_for_mma();
    }
  }

teardown:
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, TMEM_COLS);
  }
}

}  // namespace

int tc128_smem_bytes() { return static_cast<int>(SMEM_BYTES); }

cudaError_t launch_ns_tc128(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                            const NSArgs& ns, const StepArgs& st, uint64_t wait_ns, int* err,
                            int num_sms, cudaStream_t stream) {
  const int64_t ntiles = tile_end - tile_begin;
  if (ntiles <= 0) return cudaSuccess;
  const int64_t grid64 = std::min<int64_t>(ntiles, 2LL * num_sms);
  const dim3 grid(static_cast<unsigned>(grid64));
  if (st.enabled) {
    cudaFuncSetAttribute(ns_tc128_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SMEM_BYTES);
    ns_tc128_kernel<true><<<grid, NTHR, SMEM_BYTES, stream>>>(descs, ndesc, tile_begin, tile_end,
                                                              ns, st, wait_ns, err);
  } else {
    cudaFuncSetAttribute(ns_tc128_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SMEM_BYTES);
    ns_tc128_kernel<false><<<grid, NTHR, SMEM_BYTES, stream>>>(descs, ndesc, tile_begin, tile_end,
                                                               ns, st, wait_ns, err);
  }
  return cudaGetLastError();
}

}  // namespace himuon
