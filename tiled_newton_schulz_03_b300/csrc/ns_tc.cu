// Tiled Newton-Schulz on tcgen05 tensor cores, T in {64, 128}: warp-specialised,
// two tile slots per SM, TMA-fed.
//
// Method ("Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
// Optimization", abstract, sentences 3-5): every T x T tile X of a
// momentum-gradient matrix is normalised and iterated K times with
//   A = X X^T,  B = b A + c A^2,  X <- a X + B X,
// independently of every other tile. The three products per step are dense
// T x T x T contractions, run here as tcgen05.mma (bf16 operands, fp32
// accumulation in tensor memory).
//
// CTA (one per SM, 20 warps = 5 per scheduler, so 96 registers per thread):
//   warps 0-3   loader: brings the next stage's G (and M) into a staging buffer
//               with TMA, and stores the previous stage's updated momentum back
//               with TMA. Rows TMA cannot describe come in as 16-byte cp.async
//               copies of their 16-byte aligned covers (or plain loads), and
//               for those the loader applies momentum itself. Warp 0 also
//               allocates and frees tensor memory.
//   warps 4-11  slot 0, warps 12-19 slot 1 (8 warps each: lane quarter =
//               warp % 4, column half = (warp - first) / 4). A slot's warps apply
//               momentum to TMA-staged tiles, sum the squares for the
//               normalisation, run the epilogue of each product, and one thread
//               issues the slot's next product.
// The two slots hold two independent stages; while the tensor core runs one
// slot's product, the other slot's warps run their epilogue, so the serial
// chain of a tile's 3K products never leaves the tensor pipe idle for long.
//
// A stage is 128 rows: one 128 x 128 tile, or two 64 x 64 tiles stacked
// vertically (T = 64). With stacked tiles, tile t's products use the whole
// 128-row stack as the A operand and tile t's rows as the B operand; only the
// accumulator lanes of tile t are kept (the others hold unused cross products).
//
// Per slot, on chip for all K steps:
//   sX  (smem 32 KB)   X in bf16, 128-byte swizzled, 128-byte rows: operand of
//                      X X^T (K-major) and of C X (MN-major).
//   sC  (smem 32 KB)   A in bf16 (operand of A A), then C in bf16 (operand of C X).
//   R_A (TMEM, 128 columns)  accumulator of X X^T, then of A_bf A_bf onto the
//                      preload (b / c) A_bf + (e / c) I, so that C = c R_A.
//   R_X (TMEM, 128 columns)  fp32 iterate: holds a X - e X_bf before C X_bf is
//                      accumulated onto it, X' afterwards.
// Rounding: with e = a - min(a, 1.5) and C = B + e I,
//   X' = C X_bf + (a X - e X_bf) = a X + B X_bf      (exact identity),
// so X keeps fp32 precision in the a X term, and the bf16 operand C has its
// spectrum (about [-2.8, 0] for the quintic's B) centred near zero, which keeps
// its rounding small where a + B nearly cancels (rank-1 tiles).
// Weight update (step): bf16 W without decay gets D = bf16(-lr s X') added at
// L2, by a TMA reduce-add for 16-byte aligned rows or by row-wise bulk
// reduce-adds of each row's aligned interior (plus atomic adds of the ends);
// fp32 W and weight decay take a read-modify-write row pass.
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

constexpr int NWARPS = 20;
constexpr int NTHREADS = NWARPS * 32;
constexpr int SLOT_WARP0 = 4;
constexpr int LOADER_THREADS = 128;
constexpr int SLOT_THREADS = 256;

// shared memory (offsets from the 1024-byte aligned base)
// slot s: sX at s * 64 KB, sC at s * 64 KB + 32 KB
__host__ __device__ constexpr uint32_t sm_x(int s) { return static_cast<uint32_t>(s) * 65536u; }
__host__ __device__ constexpr uint32_t sm_c(int s) { return static_cast<uint32_t>(s) * 65536u + 32768u; }
constexpr uint32_t SM_S0 = 131072;  // 64 KB: fp32 tile, 4 blocks of 128 rows x 32 columns
constexpr uint32_t SM_S1 = 196608;  // 32 KB: bf16 tile, 2 blocks of 128 rows x 64 columns
constexpr uint32_t SM_END = 229376;
constexpr uint32_t SMEM_DYN = SM_END + 1024;
constexpr uint32_t TMEM_COLS = 512;

// how a sub-tile sits in the staging buffer
enum : int { FMT_U32 = 0, FMT_G16 = 1, FMT_G16M32 = 2 };

struct Ctl {
  uint64_t acc_full[2];   // tensor core -> slot: the slot's last product is complete
  uint64_t st_full[2];    // loader -> slots: staging holds stage g (barrier g % 2)
  uint64_t st_empty;      // slot -> loader: staging has been read
  uint64_t st_loaded;     // TMA -> loader: staging bytes have landed
  uint64_t drain[2];      // slot issuer: all its MMAs complete (abort path)
  uint32_t tmem_base;
  int abort_flag;
  float part[2][8];       // per slot warp: sum of squares of its row segments
  int info_mi[4], info_i0[4], info_j0[4], info_h[4], info_w[4], info_fmt[4];
  float info_s[4];
  int ticket;             // next stage to hand to a free slot
  int ticket_s[2];        // the stage each slot took
  // per slot and stacked tile, copied from info_* when the slot takes a stage:
  // how the step's weight update is written (fin_mode: 0 by the epilogue
  // threads, 1 TMA reduce-add of -lr s O, 2 row pass from sC, 3 bulk
  // reduce-add of each row's 16-byte aligned interior), matrix, origin and extent
  int fin_mode[2][2], fin_mi[2][2], fin_i0[2][2], fin_j0[2][2], fin_h[2][2], fin_w[2][2];
};

// Tile of a launch's flat list: matrix, origin and valid extent.
struct TileRef {
  int mi, i0, j0, h, w;
};
template <int T>
__device__ __forceinline__ TileRef tile_ref(const MatDesc* descs, int ndesc, int64_t tile) {
  TileRef t;
  t.mi = find_matrix(descs, ndesc, tile);
  const MatDesc& d = descs[t.mi];
  const int64_t lt = tile - d.tile_start;
  t.i0 = static_cast<int>(lt / d.tiles_w) * T;
  t.j0 = static_cast<int>(lt % d.tiles_w) * T;
  t.h = min(T, d.H - t.i0);
  t.w = min(T, d.W - t.j0);
  return t;
}

template <bool STEP>
__device__ __forceinline__ int tile_format(int flags) {
  if (!(flags & F_TMA)) return FMT_U32;
  if (STEP) return FMT_G16M32;
  return (flags & F_IN_FP32) ? FMT_U32 : FMT_G16;
}

// Output of the stage's row-pass tiles from O staged in sC (fp32, the swizzled
// layout of 4-column chunks, stage rows x 64 columns starting at tile column
// col0): out = O (NS map) or W <- wd W - lr s O (step). Warp ws of the slot
// takes stage rows [16 ws, 16 ws + 16), four at a time; lane l takes columns l
// and l + 32, so that an access touches one or two cache lines whatever the
// alignment of the rows.
template <int T, bool STEP>
__device__ __forceinline__ void w_row_pass(const Ctl& ctl, int s, const MatDesc* descs, uint32_t sc,
                                           int col0, int ws, int lane, float wd_factor) {
#pragma unroll 1
  for (int r0 = 16 * ws; r0 < 16 * ws + 16; r0 += 4) {
    float wv[4][2];
    int64_t idx[4][2];
    bool ok[4][2];
    const MatDesc* d[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int r = r0 + rr, u = r / T, rl = r % T;
      const bool row = ctl.fin_mode[s][u] == 2 && rl < ctl.fin_h[s][u];
      d[rr] = &descs[row ? ctl.fin_mi[s][u] : 0];
      const bool out32 = d[rr]->flags & F_OUT_FP32;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = col0 + lane + 32 * q;
        ok[rr][q] = row && c < ctl.fin_w[s][u];
        idx[rr][q] = static_cast<int64_t>(ctl.fin_i0[s][u] + rl) * d[rr]->ld_out + ctl.fin_j0[s][u] + c;
        wv[rr][q] = (STEP && ok[rr][q]) ? ld_val(d[rr]->out, idx[rr][q], out32) : 0.f;
      }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const bool out32 = d[rr]->flags & F_OUT_FP32;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (!ok[rr][q]) continue;
        const float o = f32_at(sc, r0 + rr, lane + 32 * q);
        st_val(d[rr]->out, idx[rr][q], out32,
               STEP ? fmaf(-d[rr]->upd_scale, o, wv[rr][q] * wd_factor) : o);
      }
    }
  }
}

// One thread adds the stage's -lr s O tiles (bf16, in the slot's sC buffer, the
// swizzled layout of the TMA box) to W by TMA reduce-add, one box of 64
// columns x T rows per 64 valid columns. Returns whether a bulk group was
// committed (it must finish reading sC before sC is written again).
template <int T>
__device__ __noinline__ bool issue_w_reduce(const Ctl& ctl, int s, const CUtensorMap* maps,
                                            uint32_t sc) {
  constexpr int TPS = 128 / T;
  bool any = false;
  for (int u = 0; u < TPS; ++u) {
    if (ctl.fin_mode[s][u] != 1) continue;
    const CUtensorMap* mw = maps + 3 * ctl.fin_mi[s][u] + 2;
    tensormap_acquire(mw);
    for (int b = 0; b < T / 64; ++b) {
      if (64 * b >= ctl.fin_w[s][u]) break;            // box wholly right of the matrix
      ptx::tma_reduce_add_2d(mw, sc + b * 16384 + u * T * 128, ctl.fin_j0[s][u] + 64 * b,
                             ctl.fin_i0[s][u]);
    }
    any = true;
  }
  if (any) ptx::bulk_commit();
  return any;
}

// ------------------------------------------------------------------ the kernel
template <int T, bool STEP>
__global__ void __launch_bounds__(NTHREADS, 1)
    ns_tc_kernel(const MatDesc* __restrict__ descs, const CUtensorMap* __restrict__ maps, int ndesc,
                 int64_t tile_begin, int64_t tile_end, NSArgs ns, StepArgs st, uint64_t wait_ns,
                 int* __restrict__ err) {
  constexpr int TPS = 128 / T;          // tiles per stage (stacked)
  constexpr int HALF = T / 2;           // columns per epilogue thread
  constexpr int NCH = HALF / 32;        // 32-column chunks per epilogue thread
  static_assert(T == 64 || T == 128, "T");

  extern __shared__ uint8_t smem_raw[];
  __shared__ Ctl ctl;

  const uint32_t sbase = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &ctl.abort_flag;

  const uint32_t b_acc[2] = {ptx::smem_u32(&ctl.acc_full[0]), ptx::smem_u32(&ctl.acc_full[1])};
  const uint32_t b_full[2] = {ptx::smem_u32(&ctl.st_full[0]), ptx::smem_u32(&ctl.st_full[1])};
  const uint32_t b_empty = ptx::smem_u32(&ctl.st_empty);
  const uint32_t b_loaded = ptx::smem_u32(&ctl.st_loaded);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(b_acc[s], 1);
      ptx::mbar_init(b_full[s], 1);
      ptx::mbar_init(ptx::smem_u32(&ctl.drain[s]), 1);
    }
    ptx::mbar_init(b_empty, 1);
    ptx::mbar_init(b_loaded, 1);
    ptx::fence_mbar_init();
    ctl.abort_flag = 0;
    ctl.ticket = 0;
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl.tmem_base), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = ctl.tmem_base;

  const int K = ns.K;
  const int64_t stride_tiles = static_cast<int64_t>(gridDim.x) * TPS;
  const int64_t first_tile = tile_begin + static_cast<int64_t>(blockIdx.x) * TPS;
  // e = a - min(a, 1.5): part of a I moved into the bf16 operand C = B + e I
  // (per NS step: step k uses coefficients (a_k, b_k, c_k))
  const StepCoef cf0 = step_coef(ns, 0);

  if (warp < 4) {
    // =============================================================== loader
    const int r = threadIdx.x;              // stage row
    int last_mi = -1;
    uint32_t ld_phase = 0;
    // TMA-staged momentum of the stage last handed to a slot: the slot writes
    // M <- mu M + G into the staging buffer; once it has released the buffer,
    // thread 0 stores it to HBM and waits until the store has read it.
    int pend_mi[TPS], pend_i0[TPS], pend_j0[TPS], pend_w[TPS];
#pragma unroll
    for (int u = 0; u < TPS; ++u) pend_mi[u] = -1;
    auto store_prev = [&]() {
      bool stored = false;
#pragma unroll
      for (int u = 0; u < TPS; ++u) {
        if (pend_mi[u] < 0) continue;
        if (!*abort_flag) {
          const CUtensorMap* mm = maps + 3 * pend_mi[u] + 1;
          for (int b = 0; b < T / 32; ++b) {
            if (32 * b >= pend_w[u]) break;     // box wholly right of the matrix
            ptx::tma_store_2d(mm, sbase + SM_S0 + b * 16384 + u * T * 128, pend_j0[u] + 32 * b,
                              pend_i0[u]);
          }
          stored = true;
        }
        pend_mi[u] = -1;
      }
      if (stored) {
        ptx::bulk_commit();
        ptx::bulk_wait_read0();
      }
    };
    int64_t g = 0;
    for (int64_t base = first_tile; base < tile_end; base += stride_tiles, ++g) {
      // staging free (the slot that read it has also finished its M stores)
      if (r == 0) wait_bar(b_empty, static_cast<uint32_t>((g & 1) ^ 1), wait_ns, abort_flag, err);
      named_sync(1, LOADER_THREADS);

      // which sub-tiles are valid, and where they come from
      TileRef ref[TPS];
      int fmt[TPS];
      bool any_tma = false;
#pragma unroll
      for (int u = 0; u < TPS; ++u) {
        const int64_t tile = base + u;
        if (tile < tile_end) {
          ref[u] = tile_ref<T>(descs, ndesc, tile);
          fmt[u] = tile_format<STEP>(descs[ref[u].mi].flags);
          any_tma |= (descs[ref[u].mi].flags & F_TMA) != 0;
        } else {
          ref[u] = TileRef{-1, 0, 0, 0, 0};
          fmt[u] = FMT_U32;
        }
      }

      // bf16 rows that TMA cannot describe are fetched as their 16-byte aligned
      // covers when the whole stage takes that path (no TMA tile in it; fp32
      // momentum)
      bool rows_cover = false;
      {
        bool ok = true;
#pragma unroll
        for (int u = 0; u < TPS; ++u) {
          if (ref[u].mi < 0) continue;
          const int f = descs[ref[u].mi].flags;
          if ((f & F_TMA) || (f & F_IN_FP32) || (STEP && (f & F_M_BF16))) ok = false;
          else rows_cover = true;
        }
        rows_cover = rows_cover && ok;
      }

      if (any_tma && r == 0 && !*abort_flag) {
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < TPS; ++u) {
          if (ref[u].mi < 0 || !(descs[ref[u].mi].flags & F_TMA)) continue;
          bytes += (fmt[u] == FMT_U32 ? 4u : 2u) * T * T;   // G: fp32 or bf16
          if (STEP) bytes += 4u * T * T;
        }
        ptx::mbar_arrive_expect_tx(b_loaded, bytes);
#pragma unroll
        for (int u = 0; u < TPS; ++u) {      // G first: its buffer holds nothing to store
          if (ref[u].mi < 0 || !(descs[ref[u].mi].flags & F_TMA)) continue;
          const CUtensorMap* mg = maps + 3 * ref[u].mi;
          if (ref[u].mi != last_mi) {
            tensormap_acquire(mg);
            if (STEP) tensormap_acquire(mg + 1);
            last_mi = ref[u].mi;
          }
          const uint32_t row_off = static_cast<uint32_t>(u * T * 128);
          if (fmt[u] == FMT_G16 || fmt[u] == FMT_G16M32) {
            for (int b = 0; b < T / 64; ++b)
              ptx::tma_load_2d(sbase + SM_S1 + b * 16384 + row_off, mg, ref[u].j0 + 64 * b,
                               ref[u].i0, b_loaded);
          } else {   // fp32 G into the fp32 tile
            for (int b = 0; b < T / 32; ++b)
              ptx::tma_load_2d(sbase + SM_S0 + b * 16384 + row_off, mg, ref[u].j0 + 32 * b,
                               ref[u].i0, b_loaded);
          }
        }
        if (STEP) {
          store_prev();                       // previous stage's M, then its buffer is free
#pragma unroll
          for (int u = 0; u < TPS; ++u) {
            if (ref[u].mi < 0 || !(descs[ref[u].mi].flags & F_TMA)) continue;
            const CUtensorMap* mm = maps + 3 * ref[u].mi + 1;
            for (int b = 0; b < T / 32; ++b)
              ptx::tma_load_2d(sbase + SM_S0 + b * 16384 + u * T * 128, mm, ref[u].j0 + 32 * b,
                               ref[u].i0, b_loaded);
          }
        }
      } else if (STEP && r == 0) {
        store_prev();
      }
      named_sync(1, LOADER_THREADS);         // plain rows below overwrite the M buffer

      // ---- rows TMA does not bring: plain loads (any alignment) into the fp32
      // tile as U, momentum applied and M written back here; zeros for a stage's
      // missing tiles. A warp takes 32 stage rows (all in one tile, since
      // T >= 64) and reads each row with its lanes along the columns, so that an
      // instruction touches one or two cache lines whatever the alignment of the
      // rows. fp32 momentum goes first, all 32 rows at once, by cp.async straight
      // into the staging tile (no registers held); G follows in batches of rows
      // held in registers while the momentum lands.
      {
        const int ln = r & 31;
        const int r0 = r & ~31;                  // first stage row of this warp
        const TileRef& me = ref[r0 / T];
        const int rl0 = r0 % T;                  // its row within the tile
        constexpr int NJ = T / 32;               // columns per lane
        if (me.mi < 0) {
#pragma unroll 1
          for (int i = 0; i < 32; ++i)
#pragma unroll
            for (int j = 0; j < NJ; ++j) f32_put(sbase + SM_S0, r0 + i, ln + 32 * j, 0.f);
        } else if (!(descs[me.mi].flags & F_TMA) && !rows_cover) {
          const MatDesc& d = descs[me.mi];
          const bool in32 = d.flags & F_IN_FP32, m32 = !(d.flags & F_M_BF16);
          auto m_index = [&](int rl, int c) {
            return static_cast<int64_t>(me.i0 + rl) * d.ld_mom + me.j0 + c;
          };
          if (STEP && m32) {
#pragma unroll 1
            for (int i = 0; i < 32; ++i) {
              const int rl = rl0 + i;
#pragma unroll
              for (int j = 0; j < NJ; ++j) {
                const int c = ln + 32 * j;
                const bool ok = rl < me.h && c < me.w;
                const float* src = static_cast<const float*>(d.mom) + (ok ? m_index(rl, c) : 0);
                ptx::cp_async_4(sbase + SM_S0 + f32_off(r0 + i, c >> 2) + (c & 3) * 4, src, ok ? 4u : 0u);
              }
            }
            ptx::cp_async_commit();
          }
          constexpr int RB = 32 / NJ;            // rows of G per batch: 32 values per lane
          constexpr int RM = 16 / NJ;            // rows per batch with bf16 momentum in registers
          const bool m_regs = STEP && !m32;
#pragma unroll 1
          for (int i = 0; i < 32; i += (m_regs ? RM : RB)) {
            const int nb = m_regs ? RM : RB;
            float gv[RB][NJ], mv[RM][NJ];
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) {
              const int rl = rl0 + i + rr;
#pragma unroll
              for (int j = 0; j < NJ; ++j) {
                const int c = ln + 32 * j;
                const bool ok = rr < nb && rl < me.h && c < me.w;
                gv[rr][j] = ok ? ld_val(d.in, static_cast<int64_t>(me.i0 + rl) * d.ld_in + me.j0 + c, in32) : 0.f;
                if (rr < RM) mv[rr][j] = (m_regs && ok) ? ld_val(d.mom, m_index(rl, c), false) : 0.f;
              }
            }
            if (STEP && m32 && i == 0) {
              ptx::cp_async_wait_all();          // this lane's momentum has landed
              __syncwarp();
            }
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) {
              if (rr >= nb) break;
              const int rl = rl0 + i + rr;
#pragma unroll
              for (int j = 0; j < NJ; ++j) {
                const int c = ln + 32 * j;
                float u = gv[rr][j];
                if (STEP) {
                  const float m = m32 ? f32_at(sbase + SM_S0, r0 + i + rr, c) : mv[rr < RM ? rr : 0][j];
                  const float mn = fmaf(st.mu, m, u);
                  if (rl < me.h && c < me.w) st_val(d.mom, m_index(rl, c), m32, mn);
                  u = st.nesterov ? fmaf(st.mu, mn, u) : mn;
                }
                f32_put(sbase + SM_S0, r0 + i + rr, c, u);
              }
            }
          }
        }
      }
      if (rows_cover) {
        // Every row of G (bf16, rows not 16-byte aligned) comes in as its 16-byte
        // aligned cover (at most 15 bytes more on either side, inside the same
        // 16-byte chunks, so always mapped memory), one 16-byte cp.async per
        // lane: all 128 stage rows (T = 64) or 64 per round (T = 128) into SM_S1
        // at a stride of 2 T + 16 bytes; fp32 momentum by 4-byte cp.async into
        // the staging tile, all rows at once. The warps then read each row with
        // the lanes along the columns, apply momentum (M written back,
        // coalesced) and store U.
        constexpr int ROWB = 2 * T + 16;
        constexpr int NJ = T / 32;
        // rows per round: all 128 when their covers fit in SM_S1 (T = 64), else 64
        constexpr int RROWS = (128 * ROWB <= 32768) ? 128 : 64;
        constexpr int ROUNDS = 128 / RROWS;
        const int ln = r & 31, wl = r >> 5;
        // every stage row a warp copies and converts below lies in one tile of
        // the stage: at T = 64 warps 0-1 take the first of two stacked 64-row
        // tiles (rows 0-63), warps 2-3 the second
        static_assert(TPS == 1 || TPS == 2, "stacked tiles per stage");
        const TileRef tw_ref = (TPS == 2 && wl >= 2) ? ref[TPS - 1] : ref[0];
        const bool tw_ok = tw_ref.mi >= 0;
        const MatDesc* tw_d = descs + (tw_ok ? tw_ref.mi : 0);
        const int64_t ld_mom = tw_d->ld_mom, ld_in = tw_d->ld_in;
        float* const mom0 = (STEP && tw_ok)
                                ? static_cast<float*>(tw_d->mom) + static_cast<int64_t>(tw_ref.i0) * ld_mom + tw_ref.j0
                                : nullptr;
        const uintptr_t gin0 = reinterpret_cast<uintptr_t>(tw_d->in) +
                               (tw_ok ? 2 * (static_cast<int64_t>(tw_ref.i0) * ld_in + tw_ref.j0) : 0);
        // A warp copies and converts only its own rows (round rd: stage rows
        // RROWS rd + (RROWS / 4) wl + i), so it waits for its own copies alone.
        if (STEP && tw_ok) {
#pragma unroll
          for (int rd = 0; rd < ROUNDS; ++rd) {
#pragma unroll 4
            for (int i = 0; i < RROWS / 4; ++i) {
              const int row = RROWS * rd + (RROWS / 4) * wl + i, rl = row % T;
#pragma unroll
              for (int j = 0; j < NJ; ++j) {
                const int c = ln + 32 * j;
                const bool ok = rl < tw_ref.h && c < tw_ref.w;
                const float* src = mom0 + (ok ? static_cast<int64_t>(rl) * ld_mom + c : 0);
                ptx::cp_async_4(sbase + SM_S0 + f32_off(row, c >> 2) + (c & 3) * 4, src, ok ? 4u : 0u);
              }
            }
          }
        }
#pragma unroll 1
        for (int rd = 0; rd < ROUNDS; ++rd) {
          // the covers of this warp's rows of the round, 16 bytes per lane
          if (tw_ok && !*abort_flag) {
#pragma unroll 4
            for (int i = 0; i < RROWS / 4; ++i) {
              const int row = RROWS * rd + (RROWS / 4) * wl + i, rl = row % T;
              const uintptr_t a = gin0 + 2 * static_cast<uint64_t>(rl) * ld_in;
              const uintptr_t lo = a & ~uintptr_t(15);
              const int nck = static_cast<int>((((a + 2 * tw_ref.w + 15) & ~uintptr_t(15)) - lo) >> 4);
              if (rl < tw_ref.h && ln < nck)
                ptx::cp_async_16(sbase + SM_S1 + (row - RROWS * rd) * ROWB + 16 * ln,
                                 reinterpret_cast<const void*>(lo + 16 * ln));
            }
          }
          ptx::cp_async_commit();
          ptx::cp_async_wait_all();                      // this warp's covers (and momentum)
          __syncwarp();
#pragma unroll 4
          for (int i = 0; i < RROWS / 4; ++i) {
            if (!tw_ok) break;                            // absent tile: zero-filled above
            const int row = RROWS * rd + (RROWS / 4) * wl + i;
            const int rl = row % T;
            const bool row_ok = rl < tw_ref.h;            // padding rows of the tile: zeros
            const uint32_t rowb = sbase + SM_S1 + (row - RROWS * rd) * ROWB +
                                  static_cast<uint32_t>((gin0 + 2 * static_cast<uint64_t>(rl) * ld_in) & 15);
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              const int c = ln + 32 * j;
              float u = 0.f;
              if (row_ok && c < tw_ref.w) {
                uint16_t gb;
                asm volatile("ld.shared.u16 %0, [%1];" : "=h"(gb) : "r"(rowb + 2 * c));
                u = __uint_as_float(static_cast<uint32_t>(gb) << 16);
                if (STEP) {
                  const float mn = fmaf(st.mu, f32_at(sbase + SM_S0, row, c), u);
                  mom0[static_cast<int64_t>(rl) * ld_mom + c] = mn;
                  u = st.nesterov ? fmaf(st.mu, mn, u) : mn;
                }
              }
              f32_put(sbase + SM_S0, row, c, u);
            }
          }
          __syncwarp();                                   // this warp's covers are refilled next round
        }
      }
      if (any_tma) {
        if (r == 0) wait_bar(b_loaded, ld_phase, wait_ns, abort_flag, err);
        ld_phase ^= 1u;
      }
      named_sync(1, LOADER_THREADS);

      if (r == 0) {
#pragma unroll
        for (int u = 0; u < TPS; ++u) {
          ctl.info_mi[u] = ref[u].mi;
          ctl.info_i0[u] = ref[u].i0;
          ctl.info_j0[u] = ref[u].j0;
          ctl.info_h[u] = ref[u].h;
          ctl.info_w[u] = ref[u].w;
          ctl.info_fmt[u] = fmt[u];
          ctl.info_s[u] = (ref[u].mi >= 0 && ns.norm == NORM_MATRIX) ? descs[ref[u].mi].norm_scale : 1.f;
          if (STEP && ref[u].mi >= 0 && fmt[u] == FMT_G16M32) {
            pend_mi[u] = ref[u].mi;
            pend_i0[u] = ref[u].i0;
            pend_j0[u] = ref[u].j0;
            pend_w[u] = ref[u].w;
          }
        }
        mbar_arrive(b_full[g & 1]);
      }
    }
    if (STEP && r == 0) {
      // the last stage's momentum: wait until its slot has released the buffer
      wait_bar(b_empty, static_cast<uint32_t>((g & 1) ^ 1), wait_ns, abort_flag, err);
      store_prev();
      ptx::bulk_wait0();
    }
  } else {
    // =============================================================== epilogue slots
    const int s = (warp - SLOT_WARP0) / 8;
    const int ws = (warp - SLOT_WARP0) % 8;
    const int q = warp & 3;                 // TMEM lane quarter
    const int hh = ws >> 2;                 // column half
    const int r = 32 * q + lane;            // stage row = TMEM lane
    const int t = r / T, rl = r % T;
    const int cbase = hh * HALF;            // first tile column of this thread
    const int nch = NCH;
    const uint32_t sx = sbase + sm_x(s), sc = sbase + sm_c(s);
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t t_a = tbase + lane_off + 256u * s + t * T;           // R_A of my tile
    const uint32_t t_x = tbase + lane_off + 256u * s + 128u + t * T;    // R_X of my tile
    uint32_t acc_ph = 0;
    // the slot's polling and MMA-issuing thread, on a scheduler of its own
    // (warp 0, the loader's, is on scheduler 0)
    const int pw = 1 + s;
    const bool issuer = (ws == pw && lane == 0);
    bool issued = false;
    bool reduce_pending = false;   // issuer: a TMA reduce-add still reads sC
    bool rows_pending = false;     // a bulk reduce-add of a W row may still be in flight
    // bf16 weights without decay whose rows TMA cannot describe: the last
    // epilogue writes bf16(-lr s O) into one shared-memory line per stage row
    // (sX and sC, free after the last product) with the row's 16-byte phase,
    // one thread per row adds the row's 16-byte aligned interior to W with a
    // bulk reduce-add (at L2, no read of W into the SM), and the few elements
    // outside it are added one by one with atomic adds
    auto bulk_rows = [&](int f) {
      return STEP && !(f & F_W_TMA) && !(f & F_OUT_FP32) && st.wd_factor == 1.f;
    };
    constexpr uint32_t LROW = 2 * T + 16;   // bytes per line: the row and its phase

    // Product p of this slot (0: X X^T -> R_A; 1: A A onto R_A; 2: C X onto R_X),
    // one 128 x T x T MMA per stacked tile, completion signalled on acc_full[s].
    auto issue = [&](int p) {
      if (!issuer || *abort_flag) return;
      constexpr uint32_t IDESC_KK = ptx::idesc_bf16_f32(128, T, false, false);
      constexpr uint32_t IDESC_KM = ptx::idesc_bf16_f32(128, T, false, true);
      ptx::tc_fence_after();
      const uint32_t dcol = tbase + 256u * s + (p == 2 ? 128u : 0u);
      const uint32_t a_base = (p == 0) ? sx : sc;
#pragma unroll
      for (int u = 0; u < TPS; ++u) {
#pragma unroll
        for (int kk = 0; kk < T / 16; ++kk) {
          const uint64_t ad = ptx::sdesc_sw128(a_base + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          uint64_t bd;
          if (p == 2) {
            bd = ptx::sdesc_sw128(sx + (u * T + 16 * kk) * 128, 16384, 1024);
          } else {
            bd = ptx::sdesc_sw128(a_base + u * T * 128 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
          }
          // A A onto (b / c) A_bf + (e / c) I, C X onto a X - e X_bf
          const uint32_t accum = (p != 0 || kk > 0) ? 1u : 0u;
          ptx::umma_bf16(dcol + u * T, ad, bd, p == 2 ? IDESC_KM : IDESC_KK, accum);
        }
      }
      ptx::umma_commit(b_acc[s]);
      issued = true;
    };

    // End of the slot's work on a row segment: store the result, or apply the update.
    // A transposed tile (tr) holds the result's column rl in the thread's row.
    auto emit = [&](const MatDesc& d, int i0, int j0, int h, int w, bool tr, int c,
                    float (&o)[32]) {
      if (tr) {
        if (rl >= w) return;
        const bool out32 = d.flags & F_OUT_FP32;
        const uint64_t nls = pk2(-d.upd_scale, -d.upd_scale);
        const uint64_t wdf = pk2(st.wd_factor, st.wd_factor);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float w0 = 0.f, w1 = 0.f;
          char* p0 = gptr(d.out, d.ld_out, i0 + c + j, j0 + rl, out32);
          char* p1 = gptr(d.out, d.ld_out, i0 + c + j + 1, j0 + rl, out32);
          const bool ok0 = c + j < h, ok1 = c + j + 1 < h;
          if (STEP) {
            if (ok0) w0 = out32 ? *reinterpret_cast<float*>(p0) : __bfloat162float(*reinterpret_cast<__nv_bfloat16*>(p0));
            if (ok1) w1 = out32 ? *reinterpret_cast<float*>(p1) : __bfloat162float(*reinterpret_cast<__nv_bfloat16*>(p1));
            upk2(fma2(nls, pk2(o[j], o[j + 1]), mul2(wdf, pk2(w0, w1))), w0, w1);
          } else {
            w0 = o[j];
            w1 = o[j + 1];
          }
          if (ok0) {
            if (out32) *reinterpret_cast<float*>(p0) = w0;
            else *reinterpret_cast<__nv_bfloat16*>(p0) = __float2bfloat16_rn(w0);
          }
          if (ok1) {
            if (out32) *reinterpret_cast<float*>(p1) = w1;
            else *reinterpret_cast<__nv_bfloat16*>(p1) = __float2bfloat16_rn(w1);
          }
        }
        return;
      }
      if (rl >= h) return;
      const int n = max(0, min(32, w - c));
      if (n == 0) return;
      const bool out32 = d.flags & F_OUT_FP32;
      char* op = gptr(d.out, d.ld_out, i0 + rl, j0, out32);
      if (STEP) {
        float wv[32];
        gload32(op, c, n, out32, d.flags & F_OUT_VEC, wv);
        const uint64_t nls = pk2(-d.upd_scale, -d.upd_scale);
        const uint64_t wdf = pk2(st.wd_factor, st.wd_factor);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          uint64_t x = fma2(nls, pk2(o[j], o[j + 1]), mul2(wdf, pk2(wv[j], wv[j + 1])));
          upk2(x, wv[j], wv[j + 1]);
        }
        gstore32(op, c, n, out32, d.flags & F_OUT_VEC, wv);
      } else {
        gstore32(op, c, n, out32, d.flags & F_OUT_VEC, o);
      }
    };

    // Operands written: make them visible to the tensor core, then the slot's
    // first thread issues product p.
    auto hand_over = [&](bool smem_written, bool tmem_written, int p) {
      if (tmem_written) ptx::tmem_wait_st();
      if (smem_written) ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      named_sync(2 + s, SLOT_THREADS);
      issue(p);
    };

    // Waits for the slot's last product.
    auto wait_acc = [&]() {
      // every thread waits itself (sleeping in try_wait, no issue slots taken):
      // no barrier hop between the poller and the others
      wait_bar(b_acc[s], acc_ph, wait_ns, abort_flag, err);
      acc_ph ^= 1u;
      ptx::tc_fence_after();
    };

    // U for tile columns [c, c + 32) of this thread's row (of X^T for a
    // transposed tile). For staged G and M (FMT_G16M32), `apply` performs the
    // momentum update M <- mu M + G in the staging buffer, from where the loader
    // stores M to HBM (each element is owned by one thread); without `apply`
    // the staged M is already the updated one.
    auto read_u = [&](int fmt, bool tr, int c, bool apply, float (&y)[32]) {
      if (tr) {
        const int r0 = t * T + c;            // stage row of tile row c
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (fmt == FMT_G16) {
            y[j] = bf16_at(sbase + SM_S1, r0 + j, rl);
          } else if (fmt == FMT_G16M32) {
            const float gv = bf16_at(sbase + SM_S1, r0 + j, rl);
            float mv = f32_at(sbase + SM_S0, r0 + j, rl);
            if (apply) {
              mv = fmaf(st.mu, mv, gv);
              f32_put(sbase + SM_S0, r0 + j, rl, mv);
            }
            y[j] = st.nesterov ? fmaf(st.mu, mv, gv) : mv;
          } else {
            y[j] = f32_at(sbase + SM_S0, r0 + j, rl);
          }
        }
      } else if (fmt == FMT_G16) {
        ld_bf16_32(sbase + SM_S1, r, c, y);
      } else if (fmt == FMT_G16M32) {
        float mv[32];
        ld_bf16_32(sbase + SM_S1, r, c, y);
        ld_f32_32(sbase + SM_S0, r, c, mv);
        const uint64_t mu2 = pk2(st.mu, st.mu);
        if (apply) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            uint64_t x = fma2(mu2, pk2(mv[j], mv[j + 1]), pk2(y[j], y[j + 1]));
            upk2(x, mv[j], mv[j + 1]);
          }
          st_f32_32(sbase + SM_S0, r, c, mv);
        }
        if (st.nesterov) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            uint64_t x = fma2(mu2, pk2(mv[j], mv[j + 1]), pk2(y[j], y[j + 1]));
            upk2(x, y[j], y[j + 1]);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) y[j] = mv[j];
        }
      } else {
        ld_f32_32(sbase + SM_S0, r, c, y);
      }
    };

    // A slot that is free takes the next stage in load order (a ticket from a
    // shared counter), so whichever slot finishes first is served first. Stage
    // g is signalled on st_full[g % 2]; the two slots hold consecutive tickets,
    // so they never wait on the same barrier at different phases.
    for (;;) {
      if (issuer) ctl.ticket_s[s] = atomicAdd(&ctl.ticket, 1);
      named_sync(2 + s, SLOT_THREADS);
      const int64_t g = ctl.ticket_s[s];
      const int64_t base = first_tile + g * stride_tiles;
      if (base >= tile_end) break;
      if (issuer)
        wait_bar(b_full[g & 1], static_cast<uint32_t>((g >> 1) & 1), wait_ns, abort_flag, err);
      named_sync(2 + s, SLOT_THREADS);
      const int mi = ctl.info_mi[t];
      const int i0 = ctl.info_i0[t], j0 = ctl.info_j0[t];
      const int th = ctl.info_h[t], tw = ctl.info_w[t];
      const int fmt = ctl.info_fmt[t];
      const float s_info = ctl.info_s[t];
      // how each tile of the stage writes its weight update, copied now: the
      // loader rewrites ctl.info_* for the next stage once staging is released
      if (issuer) {
#pragma unroll
        for (int u = 0; u < TPS; ++u) {
          const int m_u = ctl.info_mi[u];
          int mode = 0;                    // transposed tiles: by the epilogue threads
          if (m_u >= 0 && ctl.info_h[u] >= ctl.info_w[u]) {
            const int f = descs[m_u].flags;
            if (STEP) mode = (f & F_W_TMA) ? 1 : bulk_rows(f) ? 3 : 2;
            else mode = (f & F_OUT_VEC) ? 0 : 2;   // unaligned output rows: row pass
          }
          ctl.fin_mode[s][u] = mode;
          ctl.fin_mi[s][u] = m_u;
          ctl.fin_i0[s][u] = ctl.info_i0[u];
          ctl.fin_j0[s][u] = ctl.info_j0[u];
          ctl.fin_h[s][u] = ctl.info_h[u];
          ctl.fin_w[s][u] = ctl.info_w[u];
        }
      }

      // ---- prologue: staging -> sX = U_bf and R_X = a U - e U_bf, with the sum
      // of squares of U for the normalisation. The input itself (exact for bf16
      // G) is the first step's operand; the normalisation factor s enters the
      // first step's fp32 epilogue values instead (A = s^2 U_bf U_bf^T, and the
      // third product yields X_1 / s), so that X_0 = s U is never rounded twice.
      // A wide tile (fewer valid rows than columns) runs transposed: X^T has the
      // same map (p(X)^T = p(X^T)), and with the short side as the Gram's side
      // the bf16 rounding of X enters B X through a projection that averages
      // it over the long side, instead of elementwise.
      const bool tr = th < tw;
      if (STEP && mi >= 0 && !tr && !(descs[mi].flags & F_W_TMA) && rl < th && cbase < tw) {
        // the weights this thread updates at the end of the tile: pull them into
        // L2 now, so that the final update does not wait on DRAM
        // (every 128-byte line the row segment touches, whatever its alignment)
        const MatDesc& d = descs[mi];
        const bool out32 = d.flags & F_OUT_FP32;
        const char* wp = gptr(d.out, d.ld_out, i0 + rl, j0 + cbase, out32);
        const int seg = HALF * (out32 ? 4 : 2);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(wp));
        if (seg > 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(wp + 128));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(wp + seg - 1));
      }
      float ssq = 0.f;
#pragma unroll 1
      for (int ch = 0; ch < nch; ++ch) {
        const int c = cbase + 32 * ch;
        float y[32];
        read_u(fmt, tr, c, true, y);
#pragma unroll
        for (int j = 0; j < 32; ++j) ssq = fmaf(y[j], y[j], ssq);
        if (K == 0) continue;
        uint32_t pkd[16];
        st_bf16_32(sx, r, c, y, pkd);
        const uint64_t a2 = pk2(cf0.a, cf0.a), ne2 = pk2(-cf0.e, -cf0.e);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint64_t x = fma2(a2, pk2(y[2 * j], y[2 * j + 1]),
                            mul2(ne2, pk2(ptx::bf16lo(pkd[j]), ptx::bf16hi(pkd[j]))));
          upk2(x, y[2 * j], y[2 * j + 1]);
        }
        ptx::tmem_st32(t_x + c, y);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
      if (lane == 0) ctl.part[s][ws] = ssq;

      // normalisation factor of this thread's tile (partials summed in a fixed order)
      auto tile_scale = [&]() -> float {
        if (ns.norm != NORM_TILE) return s_info;
        float acc = 0.f;
        // the warps holding this tile's rows: lane quarters [t T/32, (t+1) T/32), both halves
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int qq = 0; qq < T / 32; ++qq) acc += ctl.part[s][h2 * 4 + t * (T / 32) + qq];
        return 1.f / (sqrtf(acc) + ns.eps);
      };

      if (K == 0) {
        // no iteration: the output is s U, which needs the whole tile's sum of
        // squares first, so U is read a second time (momentum already applied)
        ptx::fence_proxy_async_smem();
        named_sync(2 + s, SLOT_THREADS);
        const float sc_t = tile_scale();
#pragma unroll 1
        for (int ch = 0; ch < nch; ++ch) {
          const int c = cbase + 32 * ch;
          float y[32];
          read_u(fmt, tr, c, false, y);
          scale32(y, sc_t);
          if (mi >= 0) emit(descs[mi], i0, j0, th, tw, tr, c, y);
        }
        named_sync(2 + s, SLOT_THREADS);
        if (issuer) mbar_arrive(b_empty);
        continue;
      }
      if (reduce_pending) {                // sC is rewritten after the first product
        ptx::bulk_wait_read0();
        reduce_pending = false;
      }
      ptx::tmem_wait_st();
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      named_sync(2 + s, SLOT_THREADS);
      if (issuer) mbar_arrive(b_empty);    // staging read: the loader may refill it
      issue(0);                            // -> X X^T
      const float sc_t = tile_scale();
      const float s2 = sc_t * sc_t;

#pragma unroll 1
      for (int k = 0; k < K; ++k) {
        const StepCoef cf = step_coef(ns, k);
        const float e = cf.e;
        const bool has_c = cf.has_c;
        // ---- E1: A = X X^T in R_A
        wait_acc();
        // T = 128: both 32-column chunks of the thread loaded before one wait
        float v2[NCH][32];
        if (NCH == 2) ptx::tmem_ld32x2_sync(t_a + cbase, v2[0], t_a + cbase + 32, v2[NCH - 1]);
        else ptx::tmem_ld32_sync(t_a + cbase, v2[0]);
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          const int c = cbase + 32 * ch;
          float (&v)[32] = v2[ch];
          uint32_t pkd[16];
          if (has_c) {
            if (k == 0) scale32(v, s2);              // A = s^2 U_bf U_bf^T
            st_bf16_32(sc, r, c, v, pkd);            // A_bf
            // R_A <- (b / c) A_bf + (e / c) I, onto which A A accumulates, so
            // that c R_A = c A_bf A_bf + b A_bf + e I: B is evaluated at the
            // same rounded A_bf as the product, whose rounding then enters
            // through dB/dA = b + 2 c A, small where the two terms nearly
            // cancel, instead of through 2 c A alone
            const uint64_t bc2 = pk2(cf.bc, cf.bc);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              uint64_t x = mul2(bc2, pk2(ptx::bf16lo(pkd[j]), ptx::bf16hi(pkd[j])));
              upk2(x, v[2 * j], v[2 * j + 1]);
            }
            if ((rl >> 5) == (c >> 5)) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += (j == lane) ? cf.ec : 0.f;
            }
            ptx::tmem_st32(t_a + c, v);
          } else {
            scale32(v, k == 0 ? cf.b * s2 : cf.b);   // C = b A + e I
            if ((rl >> 5) == (c >> 5)) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] += (j == lane) ? e : 0.f;
            }
            st_bf16_32(sc, r, c, v, pkd);
          }
        }
        hand_over(true, true, has_c ? 1 : 2);    // -> A A onto R_A (or C X: R_X stores done)

        if (has_c) {
          // ---- E2: R_A = A_bf A_bf + (b / c) A_bf + (e / c) I  ->  C = c R_A
          wait_acc();
          float v2[NCH][32];
          if (NCH == 2) ptx::tmem_ld32x2_sync(t_a + cbase, v2[0], t_a + cbase + 32, v2[NCH - 1]);
          else ptx::tmem_ld32_sync(t_a + cbase, v2[0]);
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            scale32(v2[ch], cf.c);
            uint32_t pkd[16];
            st_bf16_32(sc, r, cbase + 32 * ch, v2[ch], pkd);
          }
          hand_over(true, true, 2);        // -> C X (R_X stores done)
        }

        // ---- E3: R_X = X' (on the first step X_1 / s); the next step's
        // a X' - e X'_bf takes that step's coefficients
        wait_acc();
        const bool last = (k + 1 == K);
        const StepCoef cfn = step_coef(ns, last ? k : k + 1);
        // step: W += -lr s O by a TMA reduce-add from sC (bf16 W, no decay), or
        // O staged in sC (fp32, 64 columns at a time) for a row pass
        const bool w_red = STEP && last && mi >= 0 && !tr && (descs[mi].flags & F_W_TMA);
        const bool w_bulk = last && mi >= 0 && !tr && !w_red && bulk_rows(descs[mi].flags);
        const bool w_rows = last && mi >= 0 && !tr && !w_red && !w_bulk &&
                            (STEP || !(descs[mi].flags & F_OUT_VEC));
        if (!last) {
          // the next X X^T reads only X'_bf; T = 128: both chunks loaded before one wait
          {
            float v2[NCH][32];
            if (NCH == 2) ptx::tmem_ld32x2_sync(t_x + cbase, v2[0], t_x + cbase + 32, v2[NCH - 1]);
            else ptx::tmem_ld32_sync(t_x + cbase, v2[0]);
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
              if (k == 0) scale32(v2[ch], sc_t);
              uint32_t pkd[16];
              st_bf16_32(sx, r, cbase + 32 * ch, v2[ch], pkd);
            }
          }
          hand_over(true, false, 0);             // -> next X X^T
          // Off the chain, while X X^T runs: R_X = a X' - e X'_bf (the next
          // step's coefficients) for that step's C X, which is the first
          // product to read R_X; the hand-off before it waits for these stores.
          float v2[NCH][32];
          if (NCH == 2) ptx::tmem_ld32x2_sync(t_x + cbase, v2[0], t_x + cbase + 32, v2[NCH - 1]);
          else ptx::tmem_ld32_sync(t_x + cbase, v2[0]);
          const uint64_t a2 = pk2(cfn.a, cfn.a), ne2 = pk2(-cfn.e, -cfn.e);
#pragma unroll
          for (int ch = 0; ch < NCH; ++ch) {
            float (&v)[32] = v2[ch];
            if (k == 0) scale32(v, sc_t);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const uint32_t pb = ptx::pack_bf16x2(v[j], v[j + 1]);
              uint64_t x = fma2(a2, pk2(v[j], v[j + 1]), mul2(ne2, pk2(ptx::bf16lo(pb), ptx::bf16hi(pb))));
              upk2(x, v[j], v[j + 1]);
            }
            ptx::tmem_st32(t_x + cbase + 32 * ch, v);
          }
        } else {
#pragma unroll 1
          for (int ch = 0; ch < nch; ++ch) {
            const int c = cbase + 32 * ch;
            float v[32];
            ptx::tmem_ld32_sync(t_x + c, v);
            if (k == 0) scale32(v, sc_t);
            if (w_red) {
              scale32(v, -descs[mi].upd_scale);     // -lr s O, added to W by TMA below
              uint32_t pkd[16];
              st_bf16_32(sc, r, c, v, pkd);
            } else if (w_rows) {
              if (c < 64) st_f32_32(sc, r, c, v);   // columns [64, 128) in a second round
            } else if (w_bulk) {
              const MatDesc& d = descs[mi];
              const uintptr_t g0 = reinterpret_cast<uintptr_t>(gptr(d.out, d.ld_out, i0 + rl, j0, false));
              const uintptr_t ga = (g0 + 15) & ~uintptr_t(15);
              const uintptr_t gb = (g0 + 2 * static_cast<uintptr_t>(tw)) & ~uintptr_t(15);
              const uint32_t line = sbase + sm_x(s) + static_cast<uint32_t>(r) * LROW +
                                    static_cast<uint32_t>(g0 & 15);
              const float nls = -d.upd_scale;
              if (rl < th) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  const int col = c + j;
                  if (col < tw) {
                    const uint16_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(nls * v[j]));
                    const uintptr_t ge = g0 + 2 * static_cast<uintptr_t>(col);
                    if (ge >= ga && ge < gb)
                      asm volatile("st.shared.u16 [%0], %1;" ::"r"(line + 2u * col), "h"(bits) : "memory");
                    else
                      ptx::red_add_bf16(reinterpret_cast<void*>(ge), bits);
                  }
                }
              }
            } else if (mi >= 0) {
              emit(descs[mi], i0, j0, th, tw, tr, c, v);
            }
          }
        }
      }
      if (K > 0) {
        // the stage's -lr s O tiles are in sC: one thread adds them to W
        ptx::fence_proxy_async_smem();
        named_sync(2 + s, SLOT_THREADS);
        if (STEP && issuer && !*abort_flag && issue_w_reduce<T>(ctl, s, maps, sc)) reduce_pending = true;
        if (STEP && mi >= 0 && !tr && bulk_rows(descs[mi].flags) && cbase == 0 && rl < th && !*abort_flag) {
          // this row's interior, written into its line by the row's threads above
          const MatDesc& d = descs[mi];
          const uintptr_t g0 = reinterpret_cast<uintptr_t>(gptr(d.out, d.ld_out, i0 + rl, j0, false));
          const uintptr_t ga = (g0 + 15) & ~uintptr_t(15);
          const uintptr_t gb = (g0 + 2 * static_cast<uintptr_t>(tw)) & ~uintptr_t(15);
          if (gb > ga) {
            ptx::bulk_reduce_add_bf16(reinterpret_cast<void*>(ga),
                                      sbase + sm_x(s) + static_cast<uint32_t>(r) * LROW +
                                          static_cast<uint32_t>(ga - (g0 & ~uintptr_t(15))),
                                      static_cast<uint32_t>(gb - ga));
            ptx::bulk_commit();
            // the next prologue rewrites sX: wait here until the line has been
            // read (a wait at the top of the tile loop instead, where it is
            // almost never needed, slowed the aligned step by ~1 %)
            ptx::bulk_wait_read0();
            rows_pending = true;
          }
        }
        // tiles whose W is read and written here (unaligned rows, fp32 W, weight
        // decay): O is in sC (fp32, 64 columns); the slot's warps update W row by
        // row with the lanes along the columns, so that an access touches one or
        // two cache lines whatever the alignment; T = 128 takes two rounds
        bool any_rows = false;
#pragma unroll
        for (int u = 0; u < TPS; ++u) any_rows |= ctl.fin_mode[s][u] == 2;
        if (any_rows) {
          w_row_pass<T, STEP>(ctl, s, descs, sc, 0, ws, lane, st.wd_factor);
          if (T == 128) {
            named_sync(2 + s, SLOT_THREADS);        // round 0 has read sC
            if (mi >= 0 && !tr && (STEP ? !(descs[mi].flags & F_W_TMA) : !(descs[mi].flags & F_OUT_VEC)) &&
                cbase >= 64) {
#pragma unroll 1
              for (int ch = 0; ch < nch; ++ch) {
                const int c = cbase + 32 * ch;
                float v[32];
                ptx::tmem_ld32_sync(t_x + c, v);
                if (K == 1) scale32(v, sc_t);
                st_f32_32(sc, r, c - 64, v);
              }
            }
            named_sync(2 + s, SLOT_THREADS);
            w_row_pass<T, STEP>(ctl, s, descs, sc, 64, ws, lane, st.wd_factor);
          }
        }
      }
    }
    if (reduce_pending || rows_pending) ptx::bulk_wait0();   // the reduces have completed before exit

    if (issued && *abort_flag) {
      // let every MMA this slot issued finish before tensor memory is released
      const uint32_t bd = ptx::smem_u32(&ctl.drain[s]);
      ptx::umma_commit(bd);
      const uint64_t t0 = ptx::globaltimer();
      while (!ptx::mbar_try_wait(bd, 0) && ptx::globaltimer() - t0 < wait_ns) {
      }
    }
  }

  // =============================================================== teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, TMEM_COLS);
  }
}

template <int T, bool STEP>
cudaError_t launch_t(const MatDesc* descs, const CUtensorMap* maps, int ndesc, int64_t tile_begin,
                     int64_t tile_end, const NSArgs& ns, const StepArgs& st, uint64_t wait_ns,
                     int* err, int num_sms, cudaStream_t stream) {
  constexpr int TPS = 128 / T;
  const int64_t stages = (tile_end - tile_begin + TPS - 1) / TPS;
  const int grid = static_cast<int>(std::min<int64_t>(stages, num_sms));
  cudaError_t e = cudaFuncSetAttribute(ns_tc_kernel<T, STEP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_DYN);
  if (e != cudaSuccess) return e;
  ns_tc_kernel<T, STEP><<<grid, NTHREADS, SMEM_DYN, stream>>>(descs, maps, ndesc, tile_begin,
                                                              tile_end, ns, st, wait_ns, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_tc(const MatDesc* descs, const void* maps, int ndesc, int64_t tile_begin,
                         int64_t tile_end, const NSArgs& ns, const StepArgs& st, uint64_t wait_ns,
                         int* err, int num_sms, cudaStream_t stream) {
  if (tile_end <= tile_begin) return cudaSuccess;
  const CUtensorMap* m = static_cast<const CUtensorMap*>(maps);
  if (ns.T == 128)
    return st.enabled ? launch_t<128, true>(descs, m, ndesc, tile_begin, tile_end, ns, st, wait_ns, err, num_sms, stream)
                      : launch_t<128, false>(descs, m, ndesc, tile_begin, tile_end, ns, st, wait_ns, err, num_sms, stream);
  if (ns.T == 64)
    return st.enabled ? launch_t<64, true>(descs, m, ndesc, tile_begin, tile_end, ns, st, wait_ns, err, num_sms, stream)
                      : launch_t<64, false>(descs, m, ndesc, tile_begin, tile_end, ns, st, wait_ns, err, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace himuon
