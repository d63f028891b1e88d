// Tiled Newton-Schulz for 128 < T <= 256 on a CTA pair: every tile (zero-padded
// to 256 x 256) stays on chip for all K steps, its products run on tcgen05 with
// cta_group::2.
//
// Method ("Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
// Optimization", abstract, sentences 3-6): every tile X of a momentum-gradient
// matrix is normalised and iterated K times with
//   A = X X^T,  B = b_k A + c_k A^2,  X <- a_k X + B X,
// independently of all other tiles; tile-size-specific kernels run the three
// dense products per step. A 256 x 256 tile's fp32 iterate alone fills the
// tensor memory of one SM, so a cluster of two CTAs (on two SMs) holds one
// tile: CTA c owns rows [128 c, 128 c + 128) of every operand and accumulator,
// and one thread of CTA 0 issues M = 256 products that read both CTAs' shared
// memory and write both CTAs' tensor memory.
//
// Operands (CTA c, X = the tile, n-half c = columns [128 c, 128 c + 128)):
//   X X^T  A: own rows of X, K = all 256 columns; B: the same rows (N split by CTA)
//   A A^T  A and B: own rows of A_bf (A is symmetric)
//   C X    A: own rows of C_bf; B: X restricted to the own n-half, K = all 256 rows,
//          so each CTA needs the PEER's rows of its n-half: once per step each CTA
//          copies that block of its X_bf (one 32 KB bulk copy, shared memory to
//          the peer's shared memory) while X X^T runs.
// The two products' B operands sit at the same shared-memory offsets in both
// CTAs, so X_bf is kept in four 128 x 128 buffers per CTA:
//   B[c] = own rows x own half (X X^T, K-half c)  B[1-c] = own rows x other half
//   B[2+c] = own rows x own half (C X, K-half c)  B[3-c] = peer rows x own half
// Tensor memory per CTA (512 columns): R_A (256 columns) accumulates X X^T and
// A A^T; R_X (256 columns) holds the fp32 iterate a X - e X_bf onto which C X_bf
// is accumulated (the same rounding placement as the single-SM kernel).
//
// Threads per CTA: 16 warps (lane quarter = warp % 4, 64-column quarter =
// warp / 4; 4 warps per scheduler leave 128 registers per thread) run the
// prologue and the epilogues; warp 0 also allocates tensor memory, and thread 0
// of CTA 0 issues the products. The input tile is read, momentum applied and
// the output written by these threads directly from and to global memory (rows
// pulled into L2 one tile ahead); bf16 weights without decay get their update
// as row-wise bulk reduce-adds at L2 (plus atomic adds of the ragged ends),
// other weights by a read-modify-write; wide tiles (fewer rows than columns)
// are processed transposed, like the single-SM kernel.
// Hand-off per product: all threads of both CTAs meet at the cluster barrier
// (a measured ~0.2 us, against ~0.65 us for a named barrier plus a remote
// mbarrier arrival that CTA 0's issuer waits for); CTA 0's issuer then issues,
// and completion is multicast to acc_full in both CTAs. Every mbarrier wait is
// bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "tile_util.cuh"

namespace himuon {
namespace {

using namespace tile;

constexpr int PT = 256;                       // padded tile side
constexpr int NTHREADS = 512;                 // 16 warps, 4 per scheduler: 128 registers each
constexpr int BAR_LINK = 1;                   // named barrier of all NTHREADS threads
constexpr uint32_t TMEM_COLS = 512;

// dynamic shared memory (offsets from the 1024-byte aligned base)
__host__ __device__ constexpr uint32_t sm_b(int i) { return static_cast<uint32_t>(i) * 32768u; }
constexpr uint32_t SM_C = 131072;             // 128 rows x 256 columns bf16: A_bf, then C_bf
constexpr uint32_t SM_END = 196608;
constexpr uint32_t SMEM_DYN = SM_END + 1024;

struct PairCtl {
  uint64_t acc_full;     // the pair's last product is complete (multicast commit)
  uint64_t drain;        // abort path: every issued product has completed
  uint64_t peer_in;      // the peer's block of the C X operand has arrived (bulk copy)
  uint32_t tmem_base;
  int abort_flag;
  float part[16];        // per warp: sum of squares of its elements
  float part_peer;       // the peer CTA's sum (written by the peer)
};

// Contiguous copy of `bytes` from this CTA's shared memory into the shared
// memory of another CTA of the cluster (dst and bar: cluster addresses in that
// CTA; both addresses 16-byte aligned, bytes a multiple of 16); the bytes
// complete on that CTA's mbarrier.
__device__ __forceinline__ void bulk_copy_to_cta(uint32_t dst, uint32_t src, uint32_t bytes,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 16 bytes global -> shared (both 16-byte aligned); only the first src_bytes
// are read, the rest of the 16 is zero-filled.
__device__ __forceinline__ void cp_async_16z(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

template <bool STEP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    ns_pair_kernel(const MatDesc* __restrict__ descs, int ndesc, int64_t tile_begin,
                   int64_t tile_end, NSArgs ns, StepArgs st, uint64_t wait_ns,
                   int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ PairCtl ctl;

  const uint32_t sbase = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t c = ptx::cluster_ctarank();     // 0: issues the products
  const uint32_t peer = c ^ 1u;
  volatile int* abort_flag = &ctl.abort_flag;
  const uint32_t b_acc = ptx::smem_u32(&ctl.acc_full);
  const uint32_t b_drain = ptx::smem_u32(&ctl.drain);
  const uint32_t b_peer = ptx::smem_u32(&ctl.peer_in);

  if (threadIdx.x == 0) {
    ptx::mbar_init(b_acc, 1);
    ptx::mbar_init(b_drain, 1);
    ptx::mbar_init(b_peer, 1);
    ptx::fence_mbar_init();
    ctl.abort_flag = 0;
  }
  if (warp == 0) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&ctl.tmem_base), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();           // both CTAs' barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tbase = ctl.tmem_base;

  const int K = ns.K;
  const bool issuer = (c == 0 && threadIdx.x == 0);
  const int q = warp & 3;                         // TMEM lane quarter
  const int cq = warp >> 2;                       // 64-column quarter
  const int r = 32 * q + lane;                    // local row = TMEM lane
  const int xr = 128 * static_cast<int>(c) + r;   // row of the (processed) tile
  const int xc0 = 64 * cq;                        // first tile column of this thread
  const bool own = (cq >> 1) == static_cast<int>(c);
  const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
  const uint32_t t_a = tbase + lane_off;          // R_A, columns 0..255
  const uint32_t t_x = tbase + lane_off + 256u;   // R_X, columns 256..511
  const uint32_t sc = sbase + SM_C;
  // this thread's X_bf buffers: own half -> B[c] and B[2+c] (local); other half
  // -> B[1-c] (local), which is copied as a whole into B[2+c] of the peer (the
  // two buffers have the same layout)
  const uint32_t xb1 = sbase + sm_b(own ? static_cast<int>(c) : 1 - static_cast<int>(c));
  const uint32_t xb2_local = sbase + sm_b(2 + static_cast<int>(c));
  const uint32_t blk_src = sbase + sm_b(1 - static_cast<int>(c));
  const uint32_t blk_dst = ptx::mapa_shared(xb2_local, peer);
  const uint32_t b_peer_remote = ptx::mapa_shared(b_peer, peer);

  uint32_t acc_ph = 0;
  uint32_t peer_ph = 0;          // phase of peer_in (waited by thread 0 before C X)
  bool issued = false;

  // product p of the tile (0: X X^T -> R_A; 1: A A^T -> R_A; 2: C X onto R_X)
  auto issue = [&](int p) {
    if (!issuer || *abort_flag) return;
    constexpr uint32_t IDESC_KK = ptx::idesc_bf16_f32(256, 256, false, false);
    constexpr uint32_t IDESC_KM = ptx::idesc_bf16_f32(256, 256, false, true);
    ptx::tc_fence_after();
    const uint32_t dcol = tbase + (p == 2 ? 256u : 0u);
#pragma unroll
    for (int kk = 0; kk < PT / 16; ++kk) {
      uint64_t ad, bd;
      if (p == 0) {
        ad = ptx::sdesc_sw128(sbase + sm_b(kk >> 3) + ((kk & 7) >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        bd = ad;
      } else {
        ad = ptx::sdesc_sw128(sc + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        bd = (p == 1) ? ad
                      : ptx::sdesc_sw128(sbase + sm_b(2 + (kk >> 3)) + (kk & 7) * 16 * 128, 16384, 1024);
      }
      // A A onto (b / c) A_bf + (e / c) I, C X onto a X - e X_bf
      ptx::umma_bf16_pair(dcol, ad, bd, p == 2 ? IDESC_KM : IDESC_KK, (p != 0 || kk > 0) ? 1u : 0u);
    }
    ptx::umma_commit_pair_mc(b_acc, 0x3);
    issued = true;
  };

  // Hand-off after an epilogue: operands written (shared and tensor memory) ->
  // product p. All threads of both CTAs meet at the cluster barrier (release /
  // acquire at cluster scope), then CTA 0's issuer issues. Before C X, thread 0
  // of each CTA first waits until the peer's block of this CTA's C X operand
  // has arrived (copied two products earlier, so normally long done). Every
  // thread of both CTAs makes the same sequence of hand-offs (same tiles, same
  // steps), whatever the abort flag says.
  auto hand_over = [&](bool tmem_written, int p) {
    if (tmem_written) ptx::tmem_wait_st();
    if (p == 2) {
      if (threadIdx.x == 0) wait_bar(b_peer, peer_ph, wait_ns, abort_flag, err);
      peer_ph ^= 1u;
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::cluster_sync();
    issue(p);                                  // CTA 0's issuer only
  };

  // The peer block: thread 0 of each CTA arms peer_in for it (before a cluster
  // barrier), and after that barrier thread 0 of the peer copies B[1-c] of the
  // peer (its X_bf rows of this CTA's n-half, written before the barrier) into
  // B[3-c] here. The copy runs while X X^T runs (which does not read B[3-c]);
  // B[1-c] of the sender is rewritten only after the C X hand-off, by which time
  // the copy has completed.
  auto arm_peer_block = [&]() {
    if (threadIdx.x == 0) ptx::mbar_arrive_expect_tx(b_peer, sm_b(1));
  };
  auto send_peer_block = [&]() {
    if (threadIdx.x == 0) bulk_copy_to_cta(blk_dst, blk_src, sm_b(1), b_peer_remote);
  };

  // The commit that completes acc_full comes from CTA 0's issuer, multicast by
  // the tensor core; what it orders is tensor memory, which the
  // tcgen05.fence::after_thread_sync below covers, so the wait needs CTA scope only.
  auto wait_acc = [&]() {
    wait_bar(b_acc, acc_ph, wait_ns, abort_flag, err);
    acc_ph ^= 1u;
    ptx::tc_fence_after();
  };

  const int T = ns.T;
  const int64_t ncl = gridDim.x >> 1;
  // bf16 weights without decay get their update without a read of W into the
  // SM: the last epilogue writes D = bf16(-lr s O) into one shared-memory line
  // per row (with the row's 16-byte phase), one thread per row adds the row's
  // 16-byte aligned interior by a bulk reduce-add (at L2), the ends go by atomic
  // adds. The lines lie in buffers the peer never writes: B0..B2 in CTA 0, B3
  // and sC in CTA 1.
  constexpr uint32_t PLROW = 2 * PT + 16;
  const uint32_t lbase = sbase + (c == 0 ? 0u : sm_b(3));
  bool rows_pending = false;     // this thread's bulk reduce-add still reads its line
  bool rows_wait = false;        // the last tile used the lines: wait before rewriting them
#pragma unroll 1
  for (int64_t tile = tile_begin + (blockIdx.x >> 1); tile < tile_end; tile += ncl) {
    const int mi = find_matrix(descs, ndesc, tile);
    const MatDesc& d = descs[mi];
    const int64_t lt = tile - d.tile_start;
    const int i0 = static_cast<int>(lt / d.tiles_w) * T, j0 = static_cast<int>(lt % d.tiles_w) * T;
    const int h = min(T, d.H - i0), w = min(T, d.W - j0);
    const bool tr = h < w;                 // processed transposed: X = tile^T
    const int xh = tr ? w : h, xw = tr ? h : w;
    const bool in32 = d.flags & F_IN_FP32, out32 = d.flags & F_OUT_FP32;
    const bool m16 = d.flags & F_M_BF16;
    // output (or W) rows that allow 16-byte accesses: written by each thread
    // from its own row segment; otherwise staged and written coalesced by warps
    const bool vec_out = (d.flags & F_OUT_VEC) && (j0 * (out32 ? 4 : 2)) % 16 == 0;
    const bool wbulk = STEP && !tr && !out32 && st.wd_factor == 1.f;
    if (rows_wait) {                       // (the same for every thread of the CTA)
      if (rows_pending) ptx::bulk_wait_read0();
      rows_pending = false;
      rows_wait = false;
      named_sync(BAR_LINK, NTHREADS);
    }

    // ---- prologue: U (momentum applied for a step, M written back) into
    // R_X = a U - e U_bf and the X_bf buffers; sums of squares
    float ssq = 0.f;
    {
      const StepCoef cf0 = step_coef(ns, 0);
      // 32 values of U at this thread's row, tile columns [xc, xc + 32)
      auto consume = [&](int xc, float (&u)[32]) {
#pragma unroll
        for (int j = 0; j < 32; ++j) ssq = fmaf(u[j], u[j], ssq);
        uint32_t pkd[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pkd[j] = ptx::pack_bf16x2(u[2 * j], u[2 * j + 1]);
        const int cl = xc & 127;                     // column within the 128-wide buffer
#pragma unroll
        for (int qd = 0; qd < 4; ++qd)
          ptx::st_shared_v4(xb1 + bf_off(r, (cl >> 3) + qd), pkd[4 * qd], pkd[4 * qd + 1],
                            pkd[4 * qd + 2], pkd[4 * qd + 3]);
        if (own) {
#pragma unroll
          for (int qd = 0; qd < 4; ++qd)
            ptx::st_shared_v4(xb2_local + bf_off(r, (cl >> 3) + qd), pkd[4 * qd], pkd[4 * qd + 1],
                              pkd[4 * qd + 2], pkd[4 * qd + 3]);
        }                                            // the peer's block after the first hand-off
        const uint64_t a2 = pk2(cf0.a, cf0.a), ne2 = pk2(-cf0.e, -cf0.e);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint64_t x = fma2(a2, pk2(u[2 * j], u[2 * j + 1]),
                                  mul2(ne2, pk2(ptx::bf16lo(pkd[j]), ptx::bf16hi(pkd[j]))));
          upk2(x, u[2 * j], u[2 * j + 1]);
        }
        ptx::tmem_st32(t_x + xc, u);
      };
      // rows that allow 16-byte accesses of G (and M): each thread reads its own
      // row segment with vector loads; otherwise the rows are read coalesced by
      // warps and staged through sC
      const bool vec_rows = (d.flags & F_IN_VEC) && (j0 * (in32 ? 4 : 2)) % 16 == 0 &&
                            (!STEP || ((d.flags & F_M_VEC) && (j0 * (m16 ? 2 : 4)) % 16 == 0));
      if (STEP && !tr && vec_rows && !in32 && !m16) {
        // bf16 G and fp32 M, 16-byte aligned rows: one 128-column half at a time
        // all warps copy the CTA's rows of G and M with 16-byte cp.async, the
        // lanes along a row (4 and 8 cache lines per warp instruction), into
        // shared memory that nothing else uses before this tile's first hand-off:
        // M into sC, G into B[3-c], where the peer's block lands only after that
        // hand-off. Chunk k of stage row q sits at chunk k ^ (q % 8), so the
        // per-row reads below are conflict-free. Each thread then applies
        // momentum to its row's 64 columns and puts M back in place, and the
        // warps write M back to global memory row by row, coalesced. Positions
        // outside the tile are zero-filled by the copies and not written back.
        const uint32_t stg_g = sbase + sm_b(3 - static_cast<int>(c));   // 128 rows x 256 B
        const uint32_t stg_m = sc;                                       // 128 rows x 512 B
        const int rb = 128 * static_cast<int>(c);                        // first row of this CTA
        float* const mbase = static_cast<float*>(d.mom);
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          const int cb = 128 * h2;
#pragma unroll
          for (int k = 0; k < 4; ++k) {                  // G: 128 rows x 16 chunks
            const int id = static_cast<int>(threadIdx.x) + NTHREADS * k;
            const int q = id >> 4, ck = id & 15, col = cb + 8 * ck;
            const int nb = (rb + q < xh) ? 2 * max(0, min(8, xw - col)) : 0;
            cp_async_16z(stg_g + q * 256 + ((ck ^ (q & 7)) << 4),
                         gptr(d.in, d.ld_in, i0 + (nb ? rb + q : 0), j0 + (nb ? col : 0), false), nb);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {                  // M: 128 rows x 32 chunks
            const int id = static_cast<int>(threadIdx.x) + NTHREADS * k;
            const int q = id >> 5, ck = id & 31, col = cb + 4 * ck;
            const int nb = (rb + q < xh) ? 4 * max(0, min(4, xw - col)) : 0;
            cp_async_16z(stg_m + q * 512 + ((ck ^ (q & 7)) << 4),
                         gptr(d.mom, d.ld_mom, i0 + (nb ? rb + q : 0), j0 + (nb ? col : 0), true), nb);
          }
          ptx::cp_async_commit();
          ptx::cp_async_wait_all();
          named_sync(BAR_LINK, NTHREADS);                // every warp's copies have landed
          if ((cq >> 1) == h2) {
            const uint64_t mu2 = pk2(st.mu, st.mu);
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
              const int xc = xc0 + 32 * ch, cl = xc - cb;
              float u[32], mv[32];
#pragma unroll
              for (int qd = 0; qd < 4; ++qd) {
                const uint4 w = ptx::ld_shared_v4(stg_g + r * 256 + ((((cl >> 3) + qd) ^ (r & 7)) << 4));
                u[8 * qd + 0] = ptx::bf16lo(w.x); u[8 * qd + 1] = ptx::bf16hi(w.x);
                u[8 * qd + 2] = ptx::bf16lo(w.y); u[8 * qd + 3] = ptx::bf16hi(w.y);
                u[8 * qd + 4] = ptx::bf16lo(w.z); u[8 * qd + 5] = ptx::bf16hi(w.z);
                u[8 * qd + 6] = ptx::bf16lo(w.w); u[8 * qd + 7] = ptx::bf16hi(w.w);
              }
#pragma unroll
              for (int qd = 0; qd < 8; ++qd) {
                const uint4 w = ptx::ld_shared_v4(stg_m + r * 512 + ((((cl >> 2) + qd) ^ (r & 7)) << 4));
                mv[4 * qd + 0] = __uint_as_float(w.x); mv[4 * qd + 1] = __uint_as_float(w.y);
                mv[4 * qd + 2] = __uint_as_float(w.z); mv[4 * qd + 3] = __uint_as_float(w.w);
              }
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const uint64_t mn = fma2(mu2, pk2(mv[j], mv[j + 1]), pk2(u[j], u[j + 1]));
                upk2(mn, mv[j], mv[j + 1]);
                if (st.nesterov) upk2(fma2(mu2, mn, pk2(u[j], u[j + 1])), u[j], u[j + 1]);
                else upk2(mn, u[j], u[j + 1]);
              }
#pragma unroll
              for (int qd = 0; qd < 8; ++qd)
                ptx::st_shared_v4(stg_m + r * 512 + ((((cl >> 2) + qd) ^ (r & 7)) << 4),
                                  __float_as_uint(mv[4 * qd]), __float_as_uint(mv[4 * qd + 1]),
                                  __float_as_uint(mv[4 * qd + 2]), __float_as_uint(mv[4 * qd + 3]));
              consume(xc, u);
            }
          }
          named_sync(BAR_LINK, NTHREADS);                // the half's new M is in sC
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int id = static_cast<int>(threadIdx.x) + NTHREADS * k;
            const int q = id >> 5, ck = id & 31, col = cb + 4 * ck;
            const int nv = (rb + q < xh) ? max(0, min(4, xw - col)) : 0;
            if (nv > 0) {
              const uint4 w = ptx::ld_shared_v4(stg_m + q * 512 + ((ck ^ (q & 7)) << 4));
              float* mp = mbase + static_cast<int64_t>(i0 + rb + q) * d.ld_mom + j0 + col;
              if (nv == 4) {
                *reinterpret_cast<uint4*>(mp) = w;
              } else {
                mp[0] = __uint_as_float(w.x);
                if (nv > 1) mp[1] = __uint_as_float(w.y);
                if (nv > 2) mp[2] = __uint_as_float(w.z);
              }
            }
          }
          named_sync(BAR_LINK, NTHREADS);                // staging is refilled next half
        }
      } else if (!tr && vec_rows) {
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
          const int xc = xc0 + 32 * ch;
          const int n = (xr < xh) ? max(0, min(32, xw - xc)) : 0;
          float u[32];
          gload32(gptr(d.in, d.ld_in, i0 + xr, j0, in32), xc, n, in32, true, u);
          if (STEP) {
            char* mp = gptr(d.mom, d.ld_mom, i0 + xr, j0, !m16);
            float mv[32];
            gload32(mp, xc, n, !m16, true, mv);
            const uint64_t mu2 = pk2(st.mu, st.mu);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const uint64_t mn = fma2(mu2, pk2(mv[j], mv[j + 1]), pk2(u[j], u[j + 1]));
              upk2(mn, mv[j], mv[j + 1]);
              if (st.nesterov) upk2(fma2(mu2, mn, pk2(u[j], u[j + 1])), u[j], u[j + 1]);
              else upk2(mn, u[j], u[j + 1]);
            }
            if (n > 0) gstore32(mp, xc, n, !m16, true, mv);
          }
          consume(xc, u);
        }
      } else if (!tr) {
        // one 128-column half at a time through sC (fp32): warp w reads rows
        // [8 w, 8 w + 8) of the CTA's 128 with its lanes along the columns (an
        // access touches one or two cache lines whatever the alignment), applies
        // momentum, stages U; then each thread takes its own row's 64 columns
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll 1
          for (int i = 0; i < 8; i += 4) {
            float gv[4][4], mv[4][4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int row = 128 * static_cast<int>(c) + 8 * warp + i + rr;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int col = 128 * h2 + lane + 32 * j;
                const bool ok = row < xh && col < xw;
                const int64_t gi = static_cast<int64_t>(i0 + row) * d.ld_in + j0 + col;
                const int64_t mo = static_cast<int64_t>(i0 + row) * d.ld_mom + j0 + col;
                gv[rr][j] = ok ? ld_val(d.in, gi, in32) : 0.f;
                mv[rr][j] = (STEP && ok) ? ld_val(d.mom, mo, !m16) : 0.f;
              }
            }
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int row = 128 * static_cast<int>(c) + 8 * warp + i + rr;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int col = 128 * h2 + lane + 32 * j;
                float u = gv[rr][j];
                if (STEP) {
                  const float mn = fmaf(st.mu, mv[rr][j], u);
                  if (row < xh && col < xw)
                    st_val(d.mom, static_cast<int64_t>(i0 + row) * d.ld_mom + j0 + col, !m16, mn);
                  u = st.nesterov ? fmaf(st.mu, mn, u) : mn;
                }
                f32_put(sc, 8 * warp + i + rr, lane + 32 * j, u);
              }
            }
          }
          named_sync(BAR_LINK, NTHREADS);
          if ((cq >> 1) == h2) {
#pragma unroll 1
            for (int ch = 0; ch < 2; ++ch) {
              const int xc = xc0 + 32 * ch;
              float u[32];
              ld_f32_32(sc, r, xc - 128 * h2, u);
              consume(xc, u);
            }
          }
          named_sync(BAR_LINK, NTHREADS);            // sC is restaged or rewritten next
        }
      } else {
        // X = tile^T: element (xr, xc + j) is G[i0 + xc + j][j0 + xr]; the
        // lanes of a warp read consecutive columns of one row
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
          const int xc = xc0 + 32 * ch;
          const int n = (xr < xh) ? max(0, min(32, xw - xc)) : 0;
          float u[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float x = 0.f;
            if (j < n) {
              const int64_t gi = static_cast<int64_t>(i0 + xc + j) * d.ld_in + j0 + xr;
              x = ld_val(d.in, gi, in32);
              if (STEP) {
                const int64_t mo = static_cast<int64_t>(i0 + xc + j) * d.ld_mom + j0 + xr;
                const float mn = fmaf(st.mu, ld_val(d.mom, mo, !m16), x);
                st_val(d.mom, mo, !m16, mn);
                x = st.nesterov ? fmaf(st.mu, mn, x) : mn;
              }
            }
            u[j] = x;
          }
          consume(xc, u);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
      if (lane == 0) ctl.part[warp] = ssq;

      // the next tile's rows of this thread into L2 (G, M and W for a step)
      const int64_t nt = tile + ncl;
      if (nt < tile_end) {
        const MatDesc& dn = descs[find_matrix(descs, ndesc, nt)];
        const int64_t nlt = nt - dn.tile_start;
        const int ni0 = static_cast<int>(nlt / dn.tiles_w) * T, nj0 = static_cast<int>(nlt % dn.tiles_w) * T;
        const int nh = min(T, dn.H - ni0), nw = min(T, dn.W - nj0);
        if (nh >= nw && xr < nh && xc0 < nw) {
          const bool n32 = dn.flags & F_IN_FP32;
          asm volatile("prefetch.global.L2 [%0];" ::"l"(gptr(dn.in, dn.ld_in, ni0 + xr, nj0 + xc0, n32)));
          if (STEP) {
            const bool nm32 = !(dn.flags & F_M_BF16), nw32 = dn.flags & F_OUT_FP32;
            const char* mp = gptr(dn.mom, dn.ld_mom, ni0 + xr, nj0 + xc0, nm32);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(mp));
            if (nm32) asm volatile("prefetch.global.L2 [%0];" ::"l"(mp + 128));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(gptr(dn.out, dn.ld_out, ni0 + xr, nj0 + xc0, nw32)));
          }
        }
      }
    }
    ptx::tmem_wait_st();
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    named_sync(BAR_LINK, NTHREADS);
    // tile norm: each CTA's sum (fixed order) goes to the peer; the cluster
    // barrier after it is also the hand-off of the prologue's operands
    float part_self = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) part_self += ctl.part[i];
    if (threadIdx.x == 0)
      ptx::st_cluster_f32(ptx::mapa_shared(ptx::smem_u32(&ctl.part_peer), peer), part_self);
    arm_peer_block();
    ptx::cluster_sync();
    const float tot = (c == 0) ? part_self + ctl.part_peer : ctl.part_peer + part_self;
    float sc_t = 1.f;
    if (ns.norm == NORM_TILE) sc_t = 1.f / (sqrtf(tot) + ns.eps);
    else if (ns.norm == NORM_MATRIX) sc_t = d.norm_scale;
    const float s2 = sc_t * sc_t;
    ptx::tc_fence_after();
    issue(0);                              // -> X X^T
    send_peer_block();                     // only C X, two products later, reads it

#pragma unroll 1
    for (int k = 0; k < K; ++k) {
      const StepCoef cf = step_coef(ns, k);
      const float e = cf.e;
      // ---- E1: A = X X^T (R_A) -> A_bf = bf16(s^2 R_A) and R_A <- (b / c) A_bf +
      // (e / c) I, onto which A A accumulates (c R_A = c A_bf A_bf + b A_bf + e I:
      // B is evaluated at the same rounded A_bf as the product); or C = b A + e I
      // when c = 0
      {
        wait_acc();
        float va[32], vb[32];                      // both 32-column chunks, one wait
        ptx::tmem_ld32x2_sync(t_a + xc0, va, t_a + xc0 + 32, vb);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int xc = xc0 + 32 * ch;
          float (&v)[32] = ch == 0 ? va : vb;
          const bool diag = (xr >> 5) == (xc >> 5);
          uint32_t pkd[16];
          if (cf.has_c) {
            if (k == 0) scale32(v, s2);
            st_bf16_32(sc, r, xc, v, pkd);
            const uint64_t bc2 = pk2(cf.bc, cf.bc);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              upk2(mul2(bc2, pk2(ptx::bf16lo(pkd[j]), ptx::bf16hi(pkd[j]))), v[2 * j], v[2 * j + 1]);
            if (diag) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += (j == lane) ? cf.ec : 0.f;
            }
            ptx::tmem_st32(t_a + xc, v);
          } else {
            scale32(v, k == 0 ? cf.b * s2 : cf.b);
            if (diag) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += (j == lane) ? e : 0.f;
            }
            st_bf16_32(sc, r, xc, v, pkd);
          }
        }
      }
      hand_over(true, cf.has_c ? 1 : 2);           // R_A preload (or, before C X, R_X) stored

      if (cf.has_c) {
        // ---- E2: R_A = A_bf A_bf^T + (b / c) A_bf + (e / c) I -> C = c R_A
        {
          wait_acc();
          float va[32], vb[32];
          ptx::tmem_ld32x2_sync(t_a + xc0, va, t_a + xc0 + 32, vb);
          scale32(va, cf.c);
          scale32(vb, cf.c);
          uint32_t pkd[16];
          st_bf16_32(sc, r, xc0, va, pkd);
          st_bf16_32(sc, r, xc0 + 32, vb, pkd);
        }
        hand_over(true, 2);                        // the R_X stores are done
      }

      // ---- E3: R_X = X' (on the first step X_1 / s): the next step's operands,
      // or the output / weight update
      const bool last = (k + 1 == K);
      {
        wait_acc();
        if (!last) {
          float va[32], vb[32];                    // both 32-column chunks, one wait
          ptx::tmem_ld32x2_sync(t_x + xc0, va, t_x + xc0 + 32, vb);
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const int xc = xc0 + 32 * ch;
            float (&v)[32] = ch == 0 ? va : vb;
            if (k == 0) scale32(v, sc_t);
            uint32_t pkd[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) pkd[j] = ptx::pack_bf16x2(v[2 * j], v[2 * j + 1]);
            const int cl = xc & 127;
#pragma unroll
            for (int qd = 0; qd < 4; ++qd)
              ptx::st_shared_v4(xb1 + bf_off(r, (cl >> 3) + qd), pkd[4 * qd], pkd[4 * qd + 1],
                                pkd[4 * qd + 2], pkd[4 * qd + 3]);
            if (own) {
#pragma unroll
              for (int qd = 0; qd < 4; ++qd)
                ptx::st_shared_v4(xb2_local + bf_off(r, (cl >> 3) + qd), pkd[4 * qd], pkd[4 * qd + 1],
                                  pkd[4 * qd + 2], pkd[4 * qd + 3]);
            }
          }                                          // peer block and R_X after the hand-off below
        }
#pragma unroll 1
        for (int ch = 0; ch < 2 && last; ++ch) {
          const int xc = xc0 + 32 * ch;
          float v[32];
          ptx::tmem_ld32_sync(t_x + xc, v);
          if (k == 0) scale32(v, sc_t);
          if (wbulk) {                               // D into the row's line, or atomic adds
            if (xr < xh) {
              const uintptr_t g0 = reinterpret_cast<uintptr_t>(gptr(d.out, d.ld_out, i0 + xr, j0, false));
              const uintptr_t ga = (g0 + 15) & ~uintptr_t(15);
              const uintptr_t gb = (g0 + 2 * static_cast<uintptr_t>(xw)) & ~uintptr_t(15);
              const uint32_t line = lbase + static_cast<uint32_t>(r) * PLROW + static_cast<uint32_t>(g0 & 15);
              const float nls = -d.upd_scale;
              if ((g0 & 15) == 0 && xc + 32 <= xw) {   // a 16-byte aligned row: all 32 inside
                uint32_t pkd[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) pkd[j] = ptx::pack_bf16x2(nls * v[2 * j], nls * v[2 * j + 1]);
#pragma unroll
                for (int qd = 0; qd < 4; ++qd)
                  ptx::st_shared_v4(line + 2u * xc + 16u * qd, pkd[4 * qd], pkd[4 * qd + 1], pkd[4 * qd + 2],
                                    pkd[4 * qd + 3]);
                continue;
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int col = xc + j;
                if (col < xw) {
                  const uint16_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(nls * v[j]));
                  const uintptr_t ge = g0 + 2 * static_cast<uintptr_t>(col);
                  if (ge >= ga && ge < gb)
                    asm volatile("st.shared.u16 [%0], %1;" ::"r"(line + 2u * col), "h"(bits) : "memory");
                  else
                    ptx::red_add_bf16(reinterpret_cast<void*>(ge), bits);
                }
              }
            }
            continue;
          }
          // last step. A transposed tile: out = X'^T (NS map), or W <- wd W -
          // lr s X'^T (step), the lanes writing consecutive columns of one row.
          if (!tr && vec_out) {                      // 16-byte stores of the own row segment
            const int n = (xr < xh) ? max(0, min(32, xw - xc)) : 0;
            if (n == 0) continue;
            char* op = gptr(d.out, d.ld_out, i0 + xr, j0, out32);
            if (STEP) {
              float wv[32];
              gload32(op, xc, n, out32, true, wv);
              const uint64_t nls = pk2(-d.upd_scale, -d.upd_scale), wdf = pk2(st.wd_factor, st.wd_factor);
#pragma unroll
              for (int j = 0; j < 32; j += 2)
                upk2(fma2(nls, pk2(v[j], v[j + 1]), mul2(wdf, pk2(wv[j], wv[j + 1]))), wv[j], wv[j + 1]);
              gstore32(op, xc, n, out32, true, wv);
            } else {
              gstore32(op, xc, n, out32, true, v);
            }
            continue;
          }
          if (!tr) {                                 // staged one half at a time below:
            if ((cq >> 1) == 0) st_f32_32(sc, r, xc & 127, v);   // the first half now
            continue;
          }
          const int n = (xr < xh) ? max(0, min(32, xw - xc)) : 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j >= n) break;
            const int64_t oi = static_cast<int64_t>(i0 + xc + j) * d.ld_out + j0 + xr;
            float o = v[j];
            if (STEP) o = fmaf(-d.upd_scale, o, ld_val(d.out, oi, out32) * st.wd_factor);
            st_val(d.out, oi, out32, o);
          }
        }
      }
      if (last && wbulk) {
        ptx::fence_proxy_async_smem();             // the lines, for the bulk reduce-add
        named_sync(BAR_LINK, NTHREADS);
        if (cq == 0 && xr < xh && !*abort_flag) {  // one thread per row
          const uintptr_t g0 = reinterpret_cast<uintptr_t>(gptr(d.out, d.ld_out, i0 + xr, j0, false));
          const uintptr_t ga = (g0 + 15) & ~uintptr_t(15);
          const uintptr_t gb = (g0 + 2 * static_cast<uintptr_t>(xw)) & ~uintptr_t(15);
          if (gb > ga) {
            ptx::bulk_reduce_add_bf16(reinterpret_cast<void*>(ga),
                                      lbase + static_cast<uint32_t>(r) * PLROW +
                                          static_cast<uint32_t>(ga - (g0 & ~uintptr_t(15))),
                                      static_cast<uint32_t>(gb - ga));
            ptx::bulk_commit();
            rows_pending = true;
          }
        }
        rows_wait = true;
      }
      if (last && !tr && !vec_out && !wbulk) {
        // last step, the tile as it is: X' goes through sC (fp32) one
        // 128-column half at a time (the half held by column quarters 2 h2 and
        // 2 h2 + 1 was staged above for h2 = 0); warp w then writes rows
        // [8 w, 8 w + 8) of the CTA's 128 with its lanes along the columns:
        // out = X' (NS map), or W <- wd W - lr s X' (step)
#pragma unroll 1
        for (int h2 = 0; h2 < 2; ++h2) {
          if (h2 == 1) {
            named_sync(BAR_LINK, NTHREADS);          // the first half has been written out
            if ((cq >> 1) == 1) {
#pragma unroll 1
              for (int ch = 0; ch < 2; ++ch) {
                const int xc = xc0 + 32 * ch;
                float v[32];
                ptx::tmem_ld32_sync(t_x + xc, v);
                if (K == 1) scale32(v, sc_t);
                st_f32_32(sc, r, xc & 127, v);
              }
            }
          }
          named_sync(BAR_LINK, NTHREADS);
#pragma unroll 1
          for (int i = 0; i < 8; i += 4) {
            float wv[4][4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int row = 128 * static_cast<int>(c) + 8 * warp + i + rr;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int col = 128 * h2 + lane + 32 * j;
                const int64_t oi = static_cast<int64_t>(i0 + row) * d.ld_out + j0 + col;
                wv[rr][j] = (STEP && row < xh && col < xw) ? ld_val(d.out, oi, out32) : 0.f;
              }
            }
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
              const int row = 128 * static_cast<int>(c) + 8 * warp + i + rr;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const int col = 128 * h2 + lane + 32 * j;
                if (row >= xh || col >= xw) continue;
                const int64_t oi = static_cast<int64_t>(i0 + row) * d.ld_out + j0 + col;
                float o = f32_at(sc, 8 * warp + i + rr, lane + 32 * j);
                if (STEP) o = fmaf(-d.upd_scale, o, wv[rr][j] * st.wd_factor);
                st_val(d.out, oi, out32, o);
              }
            }
          }
        }
        named_sync(BAR_LINK, NTHREADS);              // sC is free for the next tile
      }
      if (!last) {
        arm_peer_block();
        hand_over(false, 0);                       // -> next X X^T (reads X_bf only)
        send_peer_block();                         // while X X^T runs
        // Off the chain, while X X^T runs: R_X = a X' - e X'_bf (the next
        // step's coefficients) for that step's C X, the first product to read
        // R_X; the hand-off before it waits for these stores.
        const StepCoef cfn = step_coef(ns, k + 1);
        float va[32], vb[32];                      // both 32-column chunks, one wait
        ptx::tmem_ld32x2_sync(t_x + xc0, va, t_x + xc0 + 32, vb);
        const uint64_t a2 = pk2(cfn.a, cfn.a), ne2 = pk2(-cfn.e, -cfn.e);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          float (&v)[32] = ch == 0 ? va : vb;
          if (k == 0) scale32(v, sc_t);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const uint32_t pb = ptx::pack_bf16x2(v[j], v[j + 1]);
            const uint64_t x = fma2(a2, pk2(v[j], v[j + 1]), mul2(ne2, pk2(ptx::bf16lo(pb), ptx::bf16hi(pb))));
            upk2(x, v[j], v[j + 1]);
          }
          ptx::tmem_st32(t_x + xc0 + 32 * ch, v);
        }
      }
    }
  }

  if (rows_pending) ptx::bulk_wait0();           // the reduce-adds have completed
  // ---- teardown: every product this CTA issued has completed, then both CTAs
  // leave together (the peer writes into this CTA's shared memory)
  if (issued && *abort_flag) {
    ptx::umma_commit_pair_mc(b_drain, 0x1);
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(b_drain, 0) && ptx::globaltimer() - t0 < wait_ns) {
    }
  }
  // a wait for the peer block may have given up on abort: its copy lands
  // before either CTA leaves (a fresh barrier passes at once)
  if (*abort_flag && threadIdx.x == 0) (void)ptx::mbar_wait_bounded(b_peer, peer_ph ^ 1u, wait_ns);
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tbase, TMEM_COLS);
  }
}

template <bool STEP>
cudaError_t launch_p(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                     const NSArgs& ns, const StepArgs& st, uint64_t wait_ns, int* err, int num_sms,
                     cudaStream_t stream) {
  const int64_t tiles = tile_end - tile_begin;
  const int clusters = static_cast<int>(std::min<int64_t>(tiles, std::max(1, num_sms / 2)));
  cudaError_t e = cudaFuncSetAttribute(ns_pair_kernel<STEP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
  if (e != cudaSuccess) return e;
  ns_pair_kernel<STEP><<<2 * clusters, NTHREADS, SMEM_DYN, stream>>>(descs, ndesc, tile_begin,
                                                                     tile_end, ns, st, wait_ns, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_pair(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                           const NSArgs& ns, const StepArgs& st, uint64_t wait_ns, int* err,
                           int num_sms, cudaStream_t stream) {
  if (tile_end <= tile_begin) return cudaSuccess;
  if (ns.T <= 128 || ns.T > PT || ns.K < 1) return cudaErrorInvalidValue;
  return st.enabled ? launch_p<true>(descs, ndesc, tile_begin, tile_end, ns, st, wait_ns, err, num_sms, stream)
                    : launch_p<false>(descs, ndesc, tile_begin, tile_end, ns, st, wait_ns, err, num_sms, stream);
}

}  // namespace himuon
