// Internal definitions shared by the kernels and the host planner of libhimuon.
//
// A launch drains a flat list of tiles taken from several matrices (cross-layer
// batching). Each matrix is described by one MatDesc in device memory; tile
// `t` of the launch belongs to the matrix whose [tile_start, tile_start + ntiles)
// range contains it.
#pragma once

#include <cstdint>

namespace himuon {

// dtype codes, equal to himuon_dtype
enum : int32_t { DT_BF16 = 0, DT_FP32 = 1 };

// MatDesc.flags bits
enum : int32_t {
  F_IN_FP32 = 1 << 0,     // input (G) is fp32 (else bf16)
  F_OUT_FP32 = 1 << 1,    // output (out, or W for a step) is fp32 (else bf16)
  F_M_BF16 = 1 << 2,      // momentum buffer is bf16 (else fp32)
  F_IN_VEC = 1 << 3,      // 16-byte vector loads of the input are legal
  F_OUT_VEC = 1 << 4,     // 16-byte vector stores/loads of out / W are legal
  F_M_VEC = 1 << 5,       // 16-byte vector access of M is legal
  F_TMA = 1 << 6,         // tensor maps of G (and M for a step) exist: TMA staging
  F_W_TMA = 1 << 7,       // step: W (bf16, no weight decay) is updated by a TMA reduce-add
};

struct MatDesc {
  const void* in;      // G
  void* out;           // NS output, or W for a step
  void* mom;           // momentum buffer (step only)
  int64_t ld_in, ld_out, ld_mom;
  int32_t H, W;
  int32_t tiles_w;     // ceil(W / T)
  int32_t ntiles;      // ceil(H / T) * tiles_w
  int64_t tile_start;  // first tile of this matrix in the launch's flat list
  int32_t flags;
  float upd_scale;     // step: lr * s (s = per-matrix update scale)
  float norm_scale;    // NORM_MATRIX: 1 / (||G||_F + eps), written on the device
  float pad_[3];
};
static_assert(sizeof(MatDesc) == 96, "MatDesc layout");

enum : int32_t { NORM_TILE = 0, NORM_MATRIX = 1, NORM_NONE = 2 };

// One tile of the batched-GEMM path (large T): matrix, origin, valid extent,
// whether it is processed transposed (more rows than columns), and its
// normalisation factor (written on the device).
struct GTile {
  int32_t mi, i0, j0, h, w, tr;
  float s;
  float pad_;
};
static_assert(sizeof(GTile) == 32, "GTile layout");

constexpr int kMaxSteps = 64;

// NS parameters of a launch. coef[k] = (a_k, b_k, c_k) of step k, filled for
// k < K: the same triple for every step, or a per-step schedule.
struct NSArgs {
  float eps;
  int32_t norm;
  int32_t K;
  int32_t T;
  float coef[kMaxSteps][3];
};

// Coefficients of one NS step, with the shift e = a - min(a, 1.5) that the
// tensor-core kernels move from a X into the bf16 operand C = B + e I.
struct StepCoef {
  float a, b, c, e;
  float bc, ec;      // b / c and e / c (c != 0): R_A starts at (b / c) A_bf + (e / c) I
  bool has_c;        // c != 0: the step needs the product A A
};

__host__ __device__ __forceinline__ StepCoef step_coef(const NSArgs& ns, int k) {
  StepCoef s;
  s.a = ns.coef[k][0];
  s.b = ns.coef[k][1];
  s.c = ns.coef[k][2];
  s.e = s.a > 1.5f ? s.a - 1.5f : 0.f;
  s.has_c = s.c != 0.f;
  s.bc = s.has_c ? s.b / s.c : 0.f;
  s.ec = s.has_c ? s.e / s.c : 0.f;
  return s;
}

struct StepArgs {
  float mu;
  float wd_factor;     // 1 - lr * weight_decay
  int32_t nesterov;
  int32_t enabled;     // 0: plain NS launch
};

// Error codes written into the device error word (equal to himuon_status).
enum : int32_t { DEV_ERR_TIMEOUT = 4 };

// Tile -> matrix lookup by binary search over tile_start (n is small).
__device__ __forceinline__ int find_matrix(const MatDesc* __restrict__ d, int n,
                                           int64_t tile) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (d[mid].tile_start <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace himuon
