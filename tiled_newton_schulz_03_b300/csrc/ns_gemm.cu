// Large tiles and the full-matrix map on tcgen05 tensor cores, as batched GEMMs.
//
// Method ("Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
// Optimization", abstract, sentences 1-5): the same finite NS map
//   A = X X^T,  B = b A + c A^2,  X <- a X + B X
// on every tile, where a tile may be as large as the whole matrix (T >= max(H,W)
// gives the full-matrix map of Muon, sentences 1-2 and 4). A tile of this size
// does not stay on chip, so each NS step runs as three GEMM launches over all
// tiles of a batch, with the elementwise parts fused into their epilogues:
//   G1: R = X_bf X_bf^T            ->  A_bf = bf16(s^2 R)   (s only on step 0)
//   G2: R = A_bf A_bf              ->  C_bf = bf16(c R + b A_bf + e I)
//   G3: R = C_bf X_bf              ->  X' = s_0 (R + a X - e X_bf), X' in fp32
//                                      and bf16 (or the output on the last step)
// with e = a - min(a, 1.5); C X_bf + a X - e X_bf = a X + B X_bf exactly (the
// same rounding placement as the on-chip kernel). The first step's operand is
// the input itself (U_bf) and s = 1 / (||U||_F + eps) enters through s^2 and s_0.
//
// Tiles are oriented so that the Gram matrix is on the short side (a tile with
// more rows than columns is processed transposed: p(X)^T = p(X^T)) and
// zero-padded to multiples of 128 (padding stays zero through the map). A batch
// holds tiles of one padded shape (Hp <= Wp); its scratch is laid out as
// [tile][row][col] so that one 3-D TMA map covers an operand of every tile.
//
// GEMM kernel: one 128 x BN output block per CTA (BN = 256, or 128 when the
// width is not a multiple of 256 or K <= 512), K in blocks of 64 through a
// 3- or 4-stage TMA ring;
// warp 0 loads, warp 1 issues tcgen05.mma (M = 128, N = BN, K = 16), warps 2-5
// read the fp32 accumulator from TMEM (one row per thread) and run the epilogue.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace himuon {
namespace {

constexpr int GEMM_THREADS = 192;
constexpr uint32_t A_BYTES = 128 * 64 * 2;

enum : int { G_GRAM = 1, G_POLY = 2, G_APPLY = 3 };

struct GemmArgs {
  const GTile* tiles;
  const MatDesc* descs;
  int M, N, K;            // GEMM dims (same for every tile of the batch)
  int Hp, Wp;             // padded oriented tile dims
  int step;               // NS step index k
  int last;               // 1 on the last step (G3 writes the result)
  NSArgs ns;
  StepArgs st;
  uint64_t wait_ns;
  int* err;
  __nv_bfloat16* ab;      // [tile][Hp][Hp]
  __nv_bfloat16* cb;      // [tile][Hp][Hp]
  const float* x32_in;    // [tile][Hp][Wp] iterate (fp32) of this step
  const __nv_bfloat16* xb_in;
  float* x32_out;         // next iterate
  __nv_bfloat16* xb_out;
};

__device__ __forceinline__ void wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit,
                                             volatile int* abort_flag, int* err) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  uint32_t n = 0;
  while (!ptx::mbar_try_wait(bar, parity)) {
    if ((++n & 63u) == 0) {
      if (*abort_flag) return;
      if (ptx::globaltimer() - t0 > limit) {
        *abort_flag = 1;
        atomicCAS(err, 0, DEV_ERR_TIMEOUT);
        return;
      }
    }
  }
}

// Waits with a time limit only (not cut short by an abort): used where the
// waited-for asynchronous work must have finished before shared or tensor
// memory is released.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint64_t limit, int* err) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > limit) {
      atomicCAS(err, 0, DEV_ERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ void out_store(const MatDesc& d, int64_t row, int64_t col, float v) {
  const bool out32 = d.flags & F_OUT_FP32;
  char* p = static_cast<char*>(d.out) + (row * d.ld_out + col) * (out32 ? 4 : 2);
  if (out32) *reinterpret_cast<float*>(p) = v;
  else *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}
__device__ __forceinline__ float out_load(const MatDesc& d, int64_t row, int64_t col) {
  const bool out32 = d.flags & F_OUT_FP32;
  const char* p = static_cast<const char*>(d.out) + (row * d.ld_out + col) * (out32 ? 4 : 2);
  return out32 ? *reinterpret_cast<const float*>(p)
               : __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// Writes the result value of oriented element (r, c) of tile t: the output, or
// for a step the weight update W <- wd W - lr s O.
__device__ __forceinline__ void emit_elem(const GTile& t, const MatDesc& d, const StepArgs& st,
                                          int r, int c, float o) {
  const int ho = t.tr ? t.w : t.h, wo = t.tr ? t.h : t.w;
  if (r >= ho || c >= wo) return;
  const int64_t row = t.tr ? t.i0 + c : t.i0 + r;
  const int64_t col = t.tr ? t.j0 + r : t.j0 + c;
  if (st.enabled) out_store(d, row, col, fmaf(-d.upd_scale, o, out_load(d, row, col) * st.wd_factor));
  else out_store(d, row, col, o);
}

// STAGES-deep ring; small problems (K <= 512) use 128 x 128 blocks and three
// stages, so that two CTAs share an SM and one's epilogue overlaps the other's
// main loop.
template <int BN, int MODE, bool BMN, int STAGES, int MINB>
__global__ void __launch_bounds__(GEMM_THREADS, MINB)
    ns_gemm_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
                   GemmArgs g) {
  constexpr uint32_t B_BYTES = BN * 64 * 2;
  constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[STAGES], empty[STAGES], accf;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  const uint32_t sbase = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int tiles_n = g.N / BN, tiles_m = g.M / 128;
  int idx = blockIdx.x;
  const int nt = idx % tiles_n;
  idx /= tiles_n;
  const int mt = idx % tiles_m;
  const int p = idx / tiles_m;
  const int m0 = mt * 128, n0 = nt * BN;
  const int kblocks = g.K / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_u32(&accf), 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&tmem_base), BN);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = tmem_base;

  volatile int* vabort = &abort_flag;
  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % STAGES;
        if (kb >= STAGES)
          wait_bounded(ptx::smem_u32(&empty[s]), ((kb / STAGES) - 1) & 1, g.wait_ns, vabort, g.err);
        if (*vabort) break;
        issued = kb + 1;
        const uint32_t fb = ptx::smem_u32(&full[s]);
        const uint32_t sa = sbase + s * STAGE, sb = sa + A_BYTES;
        ptx::mbar_arrive_expect_tx(fb, STAGE);
        ptx::tma_load_3d(sa, &mA, kb * 64, m0, p, fb);
        if (BMN) {
          for (int i = 0; i < BN / 64; ++i)
            ptx::tma_load_3d(sb + i * 8192, &mB, n0 + 64 * i, kb * 64, p, fb);
        } else {
          ptx::tma_load_3d(sb, &mB, kb * 64, n0, p, fb);
        }
      }
      if (*vabort) {
        // every load issued must land before the CTA's shared memory goes away
        for (int kb = max(0, issued - STAGES); kb < issued; ++kb)
          wait_drain(ptx::smem_u32(&full[kb % STAGES]), (kb / STAGES) & 1, g.wait_ns, g.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = ptx::idesc_bf16_f32(128, BN, false, BMN);
      for (int kb = 0; kb < kblocks; ++kb) {
        const int s = kb % STAGES;
        wait_bounded(ptx::smem_u32(&full[s]), (kb / STAGES) & 1, g.wait_ns, vabort, g.err);
        if (*vabort) break;
        ptx::tc_fence_after();
        const uint32_t sa = sbase + s * STAGE, sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = ptx::sdesc_sw128(sa + kk * 32, 16, 1024);
          const uint64_t bd = BMN ? ptx::sdesc_sw128(sb + kk * 2048, 8192, 1024)
                                  : ptx::sdesc_sw128(sb + kk * 32, 16, 1024);
          ptx::umma_bf16(tbase, ad, bd, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::umma_commit(ptx::smem_u32(&empty[s]));
      }
      // also reached after an abort: the commit tracks every MMA issued so far
      ptx::umma_commit(ptx::smem_u32(&accf));
    }
  } else {
    // ---- epilogue: warps 2..5, TMEM lane quarter = warp % 4, one row per thread
    {
      // the global operands of this thread's row (A_bf for G2, X and X_bf for
      // G3): pulled into L2 while the main loop runs
      const int64_t rq = m0 + 32 * (warp & 3) + lane;
      if (MODE == G_POLY) {
        const char* pa = reinterpret_cast<const char*>(
            g.ab + static_cast<int64_t>(p) * g.Hp * g.Hp + rq * g.Hp + n0);
        for (int b = 0; b < BN * 2; b += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(pa + b));
      } else if (MODE == G_APPLY) {
        const int64_t o = static_cast<int64_t>(p) * g.Hp * g.Wp + rq * g.Wp + n0;
        const char* px = reinterpret_cast<const char*>(g.x32_in + o);
        const char* pb = reinterpret_cast<const char*>(g.xb_in + o);
        for (int b = 0; b < BN * 4; b += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(px + b));
        for (int b = 0; b < BN * 2; b += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(pb + b));
      }
    }
    // not cut short by an abort: every MMA must finish before TMEM is freed
    wait_drain(ptx::smem_u32(&accf), 0, g.wait_ns, g.err);
    ptx::tc_fence_after();
    const int q = warp & 3;
    const int r = m0 + 32 * q + lane;                  // oriented row within the tile
    const uint32_t taddr = tbase + (static_cast<uint32_t>(32 * q) << 16);
    const GTile& t = g.tiles[p];
    const StepCoef cf = step_coef(g.ns, g.step);       // this NS step's (a, b, c)
    const float e = cf.e;
    const int64_t hh = static_cast<int64_t>(g.Hp) * g.Hp, hw = static_cast<int64_t>(g.Hp) * g.Wp;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      const int c0 = n0 + 32 * ch;
      // G2 / G3: the chunk's global operands are requested before the TMEM
      // load, so that the two latencies overlap
      uint4 pre_b[4];
      float4 pre_x[8];
      if (MODE == G_POLY) {
        const uint4* a4 = reinterpret_cast<const uint4*>(g.ab + p * hh + static_cast<int64_t>(r) * g.Hp + c0);
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) pre_b[qd] = a4[qd];
      } else if (MODE == G_APPLY) {
        const int64_t off = p * hw + static_cast<int64_t>(r) * g.Wp + c0;
        const float4* x4 = reinterpret_cast<const float4*>(g.x32_in + off);
        const uint4* b4 = reinterpret_cast<const uint4*>(g.xb_in + off);
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) pre_b[qd] = b4[qd];
#pragma unroll
        for (int qd = 0; qd < 8; ++qd) pre_x[qd] = x4[qd];
      }
      float v[32];
      ptx::tmem_ld32_sync(taddr + 32 * ch, v);
      if (MODE == G_GRAM) {
        const float s2 = g.step == 0 ? t.s * t.s : 1.f;
        const bool has_c = cf.has_c;
        // A = s^2 R; with c = 0 there is no A A product: write C = b A + e I directly
        __nv_bfloat16* dst = (has_c ? g.ab : g.cb) + p * hh + static_cast<int64_t>(r) * g.Hp + c0;
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          float w8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float x = v[8 * qd + j] * s2;
            if (!has_c) x = x * cf.b + ((c0 + 8 * qd + j == r) ? e : 0.f);
            w8[j] = x;
          }
          d4[qd] = make_uint4(ptx::pack_bf16x2(w8[0], w8[1]), ptx::pack_bf16x2(w8[2], w8[3]),
                              ptx::pack_bf16x2(w8[4], w8[5]), ptx::pack_bf16x2(w8[6], w8[7]));
        }
      } else if (MODE == G_POLY) {
        const int64_t off = p * hh + static_cast<int64_t>(r) * g.Hp + c0;
        uint4* c4 = reinterpret_cast<uint4*>(g.cb + off);
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          const uint4 u = pre_b[qd];
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
          float w8[8];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            w8[2 * j] = fmaf(cf.c, v[8 * qd + 2 * j], cf.b * ptx::bf16lo(uw[j]));
            w8[2 * j + 1] = fmaf(cf.c, v[8 * qd + 2 * j + 1], cf.b * ptx::bf16hi(uw[j]));
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) w8[j] += (c0 + 8 * qd + j == r) ? e : 0.f;
          c4[qd] = make_uint4(ptx::pack_bf16x2(w8[0], w8[1]), ptx::pack_bf16x2(w8[2], w8[3]),
                              ptx::pack_bf16x2(w8[4], w8[5]), ptx::pack_bf16x2(w8[6], w8[7]));
        }
      } else {
        const int64_t off = p * hw + static_cast<int64_t>(r) * g.Wp + c0;
        const float sc = g.step == 0 ? t.s : 1.f;
        float o[32];
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          const uint4 u = pre_b[qd];
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
          const float4 xa = pre_x[2 * qd], xb = pre_x[2 * qd + 1];
          const float xf[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            o[8 * qd + 2 * j] =
                sc * fmaf(-e, ptx::bf16lo(uw[j]), fmaf(cf.a, xf[2 * j], v[8 * qd + 2 * j]));
            o[8 * qd + 2 * j + 1] =
                sc * fmaf(-e, ptx::bf16hi(uw[j]), fmaf(cf.a, xf[2 * j + 1], v[8 * qd + 2 * j + 1]));
          }
        }
        if (!g.last) {
          float4* y4 = reinterpret_cast<float4*>(g.x32_out + off);
          uint4* yb = reinterpret_cast<uint4*>(g.xb_out + off);
#pragma unroll
          for (int qd = 0; qd < 8; ++qd) y4[qd] = make_float4(o[4 * qd], o[4 * qd + 1], o[4 * qd + 2], o[4 * qd + 3]);
#pragma unroll
          for (int qd = 0; qd < 4; ++qd)
            yb[qd] = make_uint4(ptx::pack_bf16x2(o[8 * qd], o[8 * qd + 1]),
                                ptx::pack_bf16x2(o[8 * qd + 2], o[8 * qd + 3]),
                                ptx::pack_bf16x2(o[8 * qd + 4], o[8 * qd + 5]),
                                ptx::pack_bf16x2(o[8 * qd + 6], o[8 * qd + 7]));
        } else {
          const MatDesc& d = g.descs[t.mi];
          const int vec_mult = (d.flags & F_OUT_FP32) ? 4 : 8;   // elements per 16 bytes
          if (!t.tr && r < t.h && c0 + 32 <= t.w && (d.flags & F_OUT_VEC) &&
              (t.j0 + c0) % vec_mult == 0) {
            // a whole 32-column row segment: 16-byte accesses
            const bool out32 = d.flags & F_OUT_FP32;
            char* rowp = static_cast<char*>(d.out) +
                         (static_cast<int64_t>(t.i0 + r) * d.ld_out + t.j0 + c0) * (out32 ? 4 : 2);
            if (g.st.enabled) {
              float wv[32];
              if (out32) {
                const float4* p4 = reinterpret_cast<const float4*>(rowp);
#pragma unroll
                for (int qd = 0; qd < 8; ++qd) {
                  const float4 f = p4[qd];
                  wv[4 * qd] = f.x; wv[4 * qd + 1] = f.y; wv[4 * qd + 2] = f.z; wv[4 * qd + 3] = f.w;
                }
              } else {
                const uint4* p4 = reinterpret_cast<const uint4*>(rowp);
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                  const uint4 u = p4[qd];
                  const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    wv[8 * qd + 2 * j] = ptx::bf16lo(uw[j]);
                    wv[8 * qd + 2 * j + 1] = ptx::bf16hi(uw[j]);
                  }
                }
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = fmaf(-d.upd_scale, o[j], wv[j] * g.st.wd_factor);
            }
            if (out32) {
              float4* p4 = reinterpret_cast<float4*>(rowp);
#pragma unroll
              for (int qd = 0; qd < 8; ++qd) p4[qd] = make_float4(o[4 * qd], o[4 * qd + 1], o[4 * qd + 2], o[4 * qd + 3]);
            } else {
              uint4* p4 = reinterpret_cast<uint4*>(rowp);
#pragma unroll
              for (int qd = 0; qd < 4; ++qd)
                p4[qd] = make_uint4(ptx::pack_bf16x2(o[8 * qd], o[8 * qd + 1]),
                                    ptx::pack_bf16x2(o[8 * qd + 2], o[8 * qd + 3]),
                                    ptx::pack_bf16x2(o[8 * qd + 4], o[8 * qd + 5]),
                                    ptx::pack_bf16x2(o[8 * qd + 6], o[8 * qd + 7]));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) emit_elem(t, d, g.st, r, c0 + j, o[j]);
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, BN);
  }
}

// U of every tile (momentum applied for a step) into the oriented, padded
// fp32 and bf16 scratch, with the sum of squares of each oriented row.
// One warp per oriented row; grid (rows / 8, tiles).
template <bool STEP>
__global__ void __launch_bounds__(256) ns_gemm_gather(const GTile* __restrict__ tiles,
                                                       const MatDesc* __restrict__ descs, int Hp,
                                                       int Wp, float* __restrict__ x32,
                                                       __nv_bfloat16* __restrict__ xb,
                                                       float* __restrict__ part, StepArgs st) {
  const int p = blockIdx.y;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const GTile& t = tiles[p];
  const MatDesc& d = descs[t.mi];
  const int ho = t.tr ? t.w : t.h, wo = t.tr ? t.h : t.w;
  const bool in32 = d.flags & F_IN_FP32, m16 = d.flags & F_M_BF16;
  const int64_t base = (static_cast<int64_t>(p) * Hp + r) * Wp;
  float ss = 0.f;
  // rows of a tile that is not transposed, with 16-byte aligned source rows:
  // lane l takes 8 consecutive columns at a time (16-byte loads and stores)
  const bool vec = !t.tr && (d.flags & F_IN_VEC) && (!STEP || (d.flags & F_M_VEC)) &&
                   (t.j0 % 8 == 0);
  if (vec) {
    for (int c = 8 * lane; c < Wp; c += 256) {
      float u[8];
      if (r < ho && c + 8 <= wo) {
        const int64_t gi = static_cast<int64_t>(t.i0 + r) * d.ld_in + t.j0 + c;
        if (in32) {
          const float4* g4 = reinterpret_cast<const float4*>(static_cast<const float*>(d.in) + gi);
          const float4 a = g4[0], b = g4[1];
          u[0] = a.x; u[1] = a.y; u[2] = a.z; u[3] = a.w; u[4] = b.x; u[5] = b.y; u[6] = b.z; u[7] = b.w;
        } else {
          const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(d.in) + gi);
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            u[2 * j] = ptx::bf16lo(aw[j]);
            u[2 * j + 1] = ptx::bf16hi(aw[j]);
          }
        }
        if (STEP) {
          const int64_t mi = static_cast<int64_t>(t.i0 + r) * d.ld_mom + t.j0 + c;
          float m[8];
          if (m16) {
            const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(d.mom) + mi);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              m[2 * j] = ptx::bf16lo(aw[j]);
              m[2 * j + 1] = ptx::bf16hi(aw[j]);
            }
          } else {
            const float4* m4 = reinterpret_cast<const float4*>(static_cast<const float*>(d.mom) + mi);
            const float4 a = m4[0], b = m4[1];
            m[0] = a.x; m[1] = a.y; m[2] = a.z; m[3] = a.w; m[4] = b.x; m[5] = b.y; m[6] = b.z; m[7] = b.w;
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float mn = fmaf(st.mu, m[j], u[j]);
            u[j] = st.nesterov ? fmaf(st.mu, mn, u[j]) : mn;
            m[j] = mn;
          }
          if (m16) {
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(d.mom) + mi) =
                make_uint4(ptx::pack_bf16x2(m[0], m[1]), ptx::pack_bf16x2(m[2], m[3]),
                           ptx::pack_bf16x2(m[4], m[5]), ptx::pack_bf16x2(m[6], m[7]));
          } else {
            float4* m4 = reinterpret_cast<float4*>(static_cast<float*>(d.mom) + mi);
            m4[0] = make_float4(m[0], m[1], m[2], m[3]);
            m4[1] = make_float4(m[4], m[5], m[6], m[7]);
          }
        }
      } else {
        // the ragged edge of the tile, or padding
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x = 0.f;
          if (r < ho && c + j < wo) {
            const int64_t gi = static_cast<int64_t>(t.i0 + r) * d.ld_in + t.j0 + c + j;
            x = in32 ? static_cast<const float*>(d.in)[gi]
                     : __bfloat162float(static_cast<const __nv_bfloat16*>(d.in)[gi]);
            if (STEP) {
              const int64_t mi = static_cast<int64_t>(t.i0 + r) * d.ld_mom + t.j0 + c + j;
              const float m = m16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(d.mom)[mi])
                                  : static_cast<const float*>(d.mom)[mi];
              const float mn = fmaf(st.mu, m, x);
              if (m16) static_cast<__nv_bfloat16*>(d.mom)[mi] = __float2bfloat16_rn(mn);
              else static_cast<float*>(d.mom)[mi] = mn;
              x = st.nesterov ? fmaf(st.mu, mn, x) : mn;
            }
          }
          u[j] = x;
        }
      }
      float4* x4 = reinterpret_cast<float4*>(x32 + base + c);
      x4[0] = make_float4(u[0], u[1], u[2], u[3]);
      x4[1] = make_float4(u[4], u[5], u[6], u[7]);
      *reinterpret_cast<uint4*>(xb + base + c) =
          make_uint4(ptx::pack_bf16x2(u[0], u[1]), ptx::pack_bf16x2(u[2], u[3]),
                     ptx::pack_bf16x2(u[4], u[5]), ptx::pack_bf16x2(u[6], u[7]));
#pragma unroll
      for (int j = 0; j < 8; ++j) ss = fmaf(u[j], u[j], ss);
    }
  } else {
    for (int c = lane; c < Wp; c += 32) {
      float u = 0.f;
      if (r < ho && c < wo) {
        const int64_t row = t.tr ? t.i0 + c : t.i0 + r;
        const int64_t col = t.tr ? t.j0 + r : t.j0 + c;
        const int64_t gi = row * d.ld_in + col;
        u = in32 ? static_cast<const float*>(d.in)[gi]
                 : __bfloat162float(static_cast<const __nv_bfloat16*>(d.in)[gi]);
        if (STEP) {
          const int64_t mi = row * d.ld_mom + col;
          const float m = m16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(d.mom)[mi])
                              : static_cast<const float*>(d.mom)[mi];
          const float mn = fmaf(st.mu, m, u);
          if (m16) static_cast<__nv_bfloat16*>(d.mom)[mi] = __float2bfloat16_rn(mn);
          else static_cast<float*>(d.mom)[mi] = mn;
          u = st.nesterov ? fmaf(st.mu, mn, u) : mn;
        }
      }
      x32[base + c] = u;
      xb[base + c] = __float2bfloat16_rn(u);
      ss = fmaf(u, u, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) part[static_cast<int64_t>(p) * Hp + r] = ss;
}

// Normalisation factor of each tile, one warp per tile: lane l adds the row
// partials l, l + 32, ... in order (fp64), and the 32 lane sums are combined
// in a fixed butterfly order, so the factor does not depend on the batch.
__global__ void ns_gemm_norm(GTile* __restrict__ tiles, const MatDesc* __restrict__ descs, int n,
                             int Hp, const float* __restrict__ part, int norm, float eps) {
  const int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= n) return;                      // whole warps
  float s = 1.f;
  if (norm == NORM_TILE) {
    double acc = 0.0;
    for (int r = lane; r < Hp; r += 32) acc += part[static_cast<int64_t>(p) * Hp + r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    s = static_cast<float>(1.0 / (sqrt(acc) + static_cast<double>(eps)));
  } else if (norm == NORM_MATRIX) {
    s = descs[tiles[p].mi].norm_scale;
  }
  if (lane == 0) tiles[p].s = s;
}

// K = 0: the output is s U.
__global__ void ns_gemm_emit0(const GTile* __restrict__ tiles, const MatDesc* __restrict__ descs,
                              int Hp, int Wp, const float* __restrict__ x32, StepArgs st) {
  const int p = blockIdx.y;
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const GTile& t = tiles[p];
  const MatDesc& d = descs[t.mi];
  const int64_t base = (static_cast<int64_t>(p) * Hp + r) * Wp;
  for (int c = threadIdx.x & 31; c < Wp; c += 32) emit_elem(t, d, st, r, c, t.s * x32[base + c]);
}

template <int BN, int MODE, bool BMN, int STAGES, int MINB>
cudaError_t launch_gemm(const CUtensorMap& mA, const CUtensorMap& mB, const GemmArgs& g, int n,
                        cudaStream_t stream) {
  const uint32_t smem = STAGES * (A_BYTES + BN * 64 * 2) + 1024;
  cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel<BN, MODE, BMN, STAGES, MINB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t ctas = static_cast<int64_t>(n) * (g.M / 128) * (g.N / BN);
  ns_gemm_kernel<BN, MODE, BMN, STAGES, MINB>
      <<<static_cast<unsigned>(ctas), GEMM_THREADS, smem, stream>>>(mA, mB, g);
  return cudaGetLastError();
}

template <int MODE, bool BMN>
cudaError_t launch_gemm_bn(const CUtensorMap& mA, const CUtensorMap& mB128, const CUtensorMap& mB256,
                           const GemmArgs& g, int n, cudaStream_t stream) {
  if (g.K <= 512) return launch_gemm<128, MODE, BMN, 3, 2>(mA, mB128, g, n, stream);
  if (g.N % 256 == 0) return launch_gemm<256, MODE, BMN, 4, 1>(mA, mB256, g, n, stream);
  return launch_gemm<128, MODE, BMN, 4, 1>(mA, mB128, g, n, stream);
}

}  // namespace

int64_t gemm_scratch_bytes(int Hp, int Wp) {
  const int64_t hw = static_cast<int64_t>(Hp) * Wp, hh = static_cast<int64_t>(Hp) * Hp;
  return hw * (4 + 4 + 2 + 2) + hh * (2 + 2) + Hp * 4 + 256 * 6;
}

cudaError_t launch_ns_gemm_batch(const GTile* d_tiles, int n, int Hp, int Wp, const MatDesc* descs,
                                 const NSArgs& ns, const StepArgs& st, void* scratch,
                                 uint64_t wait_ns, int* err, cudaStream_t stream,
                                 himuon_status* status) {
  *status = HIMUON_OK;
  const int64_t hw = static_cast<int64_t>(Hp) * Wp * n, hh = static_cast<int64_t>(Hp) * Hp * n;
  auto align = [](int64_t x) { return (x + 255) & ~int64_t(255); };
  char* base = static_cast<char*>(scratch);
  int64_t off = 0;
  float* x32[2];
  __nv_bfloat16* xb[2];
  for (int i = 0; i < 2; ++i) {
    x32[i] = reinterpret_cast<float*>(base + off);
    off = align(off + hw * 4);
  }
  for (int i = 0; i < 2; ++i) {
    xb[i] = reinterpret_cast<__nv_bfloat16*>(base + off);
    off = align(off + hw * 2);
  }
  __nv_bfloat16* ab = reinterpret_cast<__nv_bfloat16*>(base + off);
  off = align(off + hh * 2);
  __nv_bfloat16* cb = reinterpret_cast<__nv_bfloat16*>(base + off);
  off = align(off + hh * 2);
  float* part = reinterpret_cast<float*>(base + off);

  GTile* tiles = const_cast<GTile*>(d_tiles);
  const dim3 rgrid(Hp / 8, n);
  if (st.enabled)
    ns_gemm_gather<true><<<rgrid, 256, 0, stream>>>(tiles, descs, Hp, Wp, x32[0], xb[0], part, st);
  else
    ns_gemm_gather<false><<<rgrid, 256, 0, stream>>>(tiles, descs, Hp, Wp, x32[0], xb[0], part, st);
  ns_gemm_norm<<<(n + 3) / 4, 128, 0, stream>>>(tiles, descs, n, Hp, part, ns.norm, ns.eps);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ns.K == 0) {
    ns_gemm_emit0<<<rgrid, 256, 0, stream>>>(tiles, descs, Hp, Wp, x32[0], st);
    return cudaGetLastError();
  }

  // 3-D maps [tile][row][col] of the operands, boxes of 64 columns
  CUtensorMap mXa[2], mXb128[2], mXb256[2], mXm[2], mAa, mAb128, mAb256, mCa;
  for (int i = 0; i < 2; ++i) {
    if (!encode_map_3d(&mXa[i], xb[i], Wp, Hp, n, 64, 128) ||
        !encode_map_3d(&mXb128[i], xb[i], Wp, Hp, n, 64, 128) ||
        !encode_map_3d(&mXb256[i], xb[i], Wp, Hp, n, 64, Hp >= 256 ? 256 : 128) ||
        !encode_map_3d(&mXm[i], xb[i], Wp, Hp, n, 64, 64)) {
      *status = HIMUON_ERR_CUDA;
      return cudaSuccess;
    }
  }
  if (!encode_map_3d(&mAa, ab, Hp, Hp, n, 64, 128) || !encode_map_3d(&mAb128, ab, Hp, Hp, n, 64, 128) ||
      !encode_map_3d(&mAb256, ab, Hp, Hp, n, 64, Hp >= 256 ? 256 : 128) ||
      !encode_map_3d(&mCa, cb, Hp, Hp, n, 64, 128)) {
    *status = HIMUON_ERR_CUDA;
    return cudaSuccess;
  }

  GemmArgs g{};
  g.tiles = d_tiles;
  g.descs = descs;
  g.Hp = Hp;
  g.Wp = Wp;
  g.ns = ns;
  g.st = st;
  g.wait_ns = wait_ns;
  g.err = err;
  g.ab = ab;
  g.cb = cb;
  for (int k = 0; k < ns.K; ++k) {
    const int cur = k & 1;
    g.step = k;
    g.last = (k + 1 == ns.K);
    g.x32_in = x32[cur];
    g.xb_in = xb[cur];
    g.x32_out = x32[cur ^ 1];
    g.xb_out = xb[cur ^ 1];
    // G1: X X^T
    g.M = Hp; g.N = Hp; g.K = Wp;
    e = launch_gemm_bn<G_GRAM, false>(mXa[cur], mXb128[cur], mXb256[cur], g, n, stream);
    if (e != cudaSuccess) return e;
    // G2: A A (steps with c = 0 have no quadratic term)
    if (step_coef(ns, k).has_c) {
      g.M = Hp; g.N = Hp; g.K = Hp;
      e = launch_gemm_bn<G_POLY, false>(mAa, mAb128, mAb256, g, n, stream);
      if (e != cudaSuccess) return e;
    }
    // G3: C X
    g.M = Hp; g.N = Wp; g.K = Hp;
    e = launch_gemm_bn<G_APPLY, true>(mCa, mXm[cur], mXm[cur], g, n, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace himuon
