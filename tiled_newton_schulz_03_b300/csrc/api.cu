// C ABI of libhimuon (declared in include/himuon.h): argument checks, the
// cross-layer work plan (flat tile list over all matrices), memory-bounded
// chunking, workspace management and kernel dispatch.
//
// Method: "Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
// Optimization", abstract: tiles are independent (sentences 3-4), so the tiles
// of any number of matrices form one work list (cross-layer batching) that can
// be cut anywhere into launches (memory-bounded chunking), and T may differ from
// call to call (runtime tile-size schedules) -- sentence 6.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "../../include/himuon.h"
#include "common.cuh"
#include "kernels.h"

using namespace himuon;

namespace {

thread_local std::string g_last_error;

himuon_status fail(himuon_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

himuon_status cuda_fail(cudaError_t e, const char* where) {
  return fail(HIMUON_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

constexpr int32_t kMaxK = kMaxSteps;
constexpr int64_t kMaxDim = (1LL << 31) - 1024;
constexpr size_t kFp32ScratchCap = size_t(512) << 20;  // bytes of fp32-path scratch per sub-batch

bool valid_dtype(int32_t t) { return t == HIMUON_BF16 || t == HIMUON_FP32; }
int64_t esize(int32_t t) { return t == HIMUON_FP32 ? 4 : 2; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p, int64_t ld, int32_t t) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * esize(t)) % 16 == 0);
}

// Byte range [lo, hi) touched by an H x W matrix with leading dimension ld.
void byte_range(const void* p, int64_t H, int64_t W, int64_t ld, int32_t t, uintptr_t* lo,
                uintptr_t* hi) {
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + static_cast<uintptr_t>(((H - 1) * ld + W) * esize(t));
}

bool overlaps(const void* a, int64_t H, int64_t W, int64_t lda, int32_t ta, const void* b,
              int64_t ldb, int32_t tb) {
  uintptr_t a0, a1, b0, b1;
  byte_range(a, H, W, lda, ta, &a0, &a1);
  byte_range(b, H, W, ldb, tb, &b0, &b1);
  return a0 < b1 && b0 < a1;
}

himuon_status check_ns_params(const himuon_ns_params& p) {
  if (!(p.norm == HIMUON_NORM_TILE || p.norm == HIMUON_NORM_MATRIX || p.norm == HIMUON_NORM_NONE))
    return fail(HIMUON_ERR_INVALID_ARG, "ns params: unknown norm mode");
  if (!(p.path == HIMUON_PATH_AUTO || p.path == HIMUON_PATH_TENSOR || p.path == HIMUON_PATH_FP32))
    return fail(HIMUON_ERR_INVALID_ARG, "ns params: unknown path");
  if (!p.step_coeffs && (!std::isfinite(p.a) || !std::isfinite(p.b) || !std::isfinite(p.c)))
    return fail(HIMUON_ERR_INVALID_ARG, "ns params: coefficients must be finite");
  if (!(p.eps >= 0.f) || !std::isfinite(p.eps))
    return fail(HIMUON_ERR_INVALID_ARG, "ns params: eps must be finite and >= 0");
  return HIMUON_OK;
}

// Kernel arguments of the NS map: the coefficients of every step (the same
// triple K times, or the caller's per-step schedule), normalisation, K and T.
himuon_status make_ns_args(const himuon_ns_params& p, int32_t K, int32_t T, NSArgs* ns) {
  std::memset(ns, 0, sizeof(NSArgs));
  ns->eps = p.eps;
  ns->norm = p.norm;
  ns->K = K;
  ns->T = T;
  for (int32_t k = 0; k < K; ++k) {
    const float* c = p.step_coeffs ? p.step_coeffs + 3 * k : nullptr;
    ns->coef[k][0] = c ? c[0] : p.a;
    ns->coef[k][1] = c ? c[1] : p.b;
    ns->coef[k][2] = c ? c[2] : p.c;
    if (!std::isfinite(ns->coef[k][0]) || !std::isfinite(ns->coef[k][1]) ||
        !std::isfinite(ns->coef[k][2]))
      return fail(HIMUON_ERR_INVALID_ARG,
                  "ns params: coefficients of step " + std::to_string(k) + " must be finite");
    // the on-chip kernels start the A A accumulator at (b / c) A_bf + (e / c) I
    const StepCoef sc = step_coef(*ns, k);
    if (sc.has_c && !(std::fabs(sc.bc) <= 1e30f && std::fabs(sc.ec) <= 1e30f))
      return fail(HIMUON_ERR_INVALID_ARG,
                  "ns params: step " + std::to_string(k) + ": c must be 0 or |b / c|, |e / c| <= 1e30");
  }
  return HIMUON_OK;
}

himuon_status check_shape(int64_t H, int64_t W, int64_t ld, const char* what) {
  if (H < 1 || W < 1) return fail(HIMUON_ERR_INVALID_ARG, std::string(what) + ": H and W must be >= 1");
  if (H > kMaxDim || W > kMaxDim) return fail(HIMUON_ERR_INVALID_ARG, std::string(what) + ": H or W too large");
  if (ld < W) return fail(HIMUON_ERR_INVALID_ARG, std::string(what) + ": leading dimension < W");
  return HIMUON_OK;
}

}  // namespace

namespace himuon {
// Lets the other translation units of the library set the last-error string.
void record_last_error(const std::string& msg) { g_last_error = msg; }
}  // namespace himuon

struct himuon_handle {
  int device = -1;
  int num_sms = 0;
  void* ws = nullptr;          // descriptor table, part offsets, norm partials
  size_t ws_bytes = 0;
  float* scratch = nullptr;    // fp32-path tile buffers
  size_t scratch_bytes = 0;
  int* d_err = nullptr;        // device error word
  void* tiles = nullptr;       // GEMM-path tile table
  size_t tiles_bytes = 0;
  uint64_t wait_ns = 2000000000ull;
  int64_t launches = 0;        // kernels launched through this handle
  std::vector<unsigned char> host;
  // The bytes the device workspace holds since the last upload: a call whose
  // plan (descriptors, offsets, tensor maps) is byte-identical -- the same
  // matrices step after step -- skips the upload. Kernels only write fields
  // that every launch recomputes (per-matrix norm factors, norm partials).
  std::vector<unsigned char> ws_image;
  // Encoded tensor maps by (address, shape, leading dimension, type, box).
  std::map<std::array<int64_t, 7>, CUtensorMap> map_cache;
};

namespace {

himuon_status grow(void** buf, size_t* have, size_t need, cudaStream_t stream, const char* what) {
  if (need <= *have) return HIMUON_OK;
  // (a new workspace holds nothing: callers that track its contents reset them)
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "workspace growth: stream sync");
  const size_t n = std::max(need, *have + *have / 2);
  if (*buf) cudaFree(*buf);
  *buf = nullptr;
  *have = 0;
  e = cudaMalloc(buf, n);
  if (e != cudaSuccess) {
    cudaGetLastError();
    *buf = nullptr;
    return fail(HIMUON_ERR_OUT_OF_MEMORY, std::string(what) + ": cudaMalloc failed");
  }
  *have = n;
  return HIMUON_OK;
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

// 2-D tiled map of an H x W row-major matrix (leading dimension ld elements),
// box of box_w columns x box_h rows, 128-byte swizzle, zero fill outside.
bool make_map(CUtensorMap* m, const void* base, int64_t H, int64_t W, int64_t ld, bool fp32,
              int box_w, int box_h) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const int64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(H)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * es)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_w), static_cast<cuuint32_t>(box_h)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// make_map through the handle's cache of encoded maps.
bool cached_map(himuon_handle* h, CUtensorMap* m, const void* base, int64_t H, int64_t W,
                int64_t ld, bool fp32, int box_w, int box_h) {
  const std::array<int64_t, 7> key{static_cast<int64_t>(reinterpret_cast<uintptr_t>(base)), H, W,
                                   ld, fp32 ? 1 : 0, box_w, box_h};
  auto it = h->map_cache.find(key);
  if (it != h->map_cache.end()) {
    *m = it->second;
    return true;
  }
  if (!make_map(m, base, H, W, ld, fp32, box_w, box_h)) return false;
  if (h->map_cache.size() >= 65536) h->map_cache.clear();
  h->map_cache.emplace(key, *m);
  return true;
}

}  // namespace

namespace himuon {
bool encode_map_3d(void* map, const void* base, int64_t C, int64_t R, int64_t n, int box_c,
                   int box_r) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(R),
                        static_cast<cuuint64_t>(n)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(C * 2), static_cast<cuuint64_t>(C * R * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_c), static_cast<cuuint32_t>(box_r), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace himuon

namespace {

himuon_status check_handle(himuon_handle* h) {
  if (!h) return fail(HIMUON_ERR_INVALID_ARG, "handle is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev != h->device)
    return fail(HIMUON_ERR_INVALID_ARG, "handle was created on another device than the current one");
  return HIMUON_OK;
}

constexpr int64_t kGemmScratchCap = int64_t(2) << 30;  // scratch bytes of one GEMM-path batch

// Large tiles and the full-matrix map: every tile becomes a chain of GEMMs.
// Tiles are oriented so that the Gram matrix is on the short side, padded to
// multiples of 128, grouped by padded shape and run in batches whose scratch
// stays within kGemmScratchCap.
himuon_status run_gemm_path(himuon_handle* h, const std::vector<MatDesc>& descs,
                            const MatDesc* d_descs, int32_t T, const NSArgs& ns,
                            const StepArgs& st,
                            const std::vector<std::pair<int64_t, int64_t>>& chunks,
                            cudaStream_t stream) {
  auto r128 = [](int64_t x) { return static_cast<int>((x + 127) / 128 * 128); };
  for (const auto& c : chunks) {
    // tiles of this chunk, grouped by padded oriented shape
    std::map<std::pair<int, int>, std::vector<GTile>> groups;
    for (size_t mi = 0; mi < descs.size(); ++mi) {
      const MatDesc& d = descs[mi];
      const int64_t lo = std::max<int64_t>(c.first, d.tile_start);
      const int64_t hi = std::min<int64_t>(c.second, d.tile_start + d.ntiles);
      for (int64_t t = lo; t < hi; ++t) {
        const int64_t lt = t - d.tile_start;
        GTile g{};
        g.mi = static_cast<int32_t>(mi);
        g.i0 = static_cast<int32_t>(lt / d.tiles_w) * T;
        g.j0 = static_cast<int32_t>(lt % d.tiles_w) * T;
        g.h = std::min<int32_t>(T, d.H - g.i0);
        g.w = std::min<int32_t>(T, d.W - g.j0);
        g.tr = g.h > g.w ? 1 : 0;
        g.s = 1.f;
        groups[{r128(std::min(g.h, g.w)), r128(std::max(g.h, g.w))}].push_back(g);
      }
    }
    for (auto& kv : groups) {
      const int Hp = kv.first.first, Wp = kv.first.second;
      const int64_t per = gemm_scratch_bytes(Hp, Wp);
      const int64_t nb = std::max<int64_t>(1, std::min<int64_t>(kGemmScratchCap / per, 1 << 20));
      const std::vector<GTile>& all = kv.second;
      for (size_t b0 = 0; b0 < all.size(); b0 += static_cast<size_t>(nb)) {
        const int nt = static_cast<int>(std::min<size_t>(static_cast<size_t>(nb), all.size() - b0));
        void* scr = h->scratch;
        himuon_status s = grow(&scr, &h->scratch_bytes, static_cast<size_t>(per * nt), stream,
                               "GEMM-path scratch");
        h->scratch = static_cast<float*>(scr);
        if (s != HIMUON_OK) return s;
        void* tl = h->tiles;
        s = grow(&tl, &h->tiles_bytes, sizeof(GTile) * nt, stream, "tile table");
        h->tiles = tl;
        if (s != HIMUON_OK) return s;
        // pageable source: staged before the call returns
        cudaError_t e = cudaMemcpyAsync(h->tiles, all.data() + b0, sizeof(GTile) * nt,
                                        cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "tile table upload");
        himuon_status ms = HIMUON_OK;
        e = launch_ns_gemm_batch(static_cast<const GTile*>(h->tiles), nt, Hp, Wp, d_descs, ns, st,
                                 h->scratch, h->wait_ns, h->d_err, stream, &ms);
        if (ms != HIMUON_OK) return fail(ms, "GEMM path: tensor map encoding failed");
        if (e != cudaSuccess) return cuda_fail(e, "GEMM path launch");
        int64_t per_step = 0;
        for (int k = 0; k < ns.K; ++k) per_step += step_coef(ns, k).has_c ? 3 : 2;
        h->launches += 2 + (ns.K == 0 ? 1 : per_step);
      }
    }
  }
  return HIMUON_OK;
}

// Runs the tiled NS map (or the fused step) over the matrices in `descs`.
himuon_status run_plan(himuon_handle* h, std::vector<MatDesc>& descs, int32_t T, int32_t K,
                       const himuon_ns_params& p, const StepArgs& st, size_t chunk_bytes,
                       cudaStream_t stream) {
  const int n = static_cast<int>(descs.size());
  if (T < 1) return fail(HIMUON_ERR_INVALID_ARG, "T must be >= 1");
  if (K < 0 || K > kMaxK) return fail(HIMUON_ERR_INVALID_ARG, "K must be in [0, 64]");

  // ---- tile list and the per-tile byte bound used for chunking
  int64_t total = 0, maxside = 0;
  std::vector<int64_t> tile_bytes(n);
  for (int i = 0; i < n; ++i) {
    MatDesc& d = descs[i];
    d.tiles_w = static_cast<int32_t>(cdiv(d.W, T));
    const int64_t nt = cdiv(d.H, T) * d.tiles_w;
    if (nt > (1LL << 31) - 1) return fail(HIMUON_ERR_INVALID_ARG, "too many tiles in one matrix");
    d.ntiles = static_cast<int32_t>(nt);
    d.tile_start = total;
    total += nt;
    maxside = std::max<int64_t>(maxside, std::max(d.H, d.W));
    int64_t per = esize((d.flags & F_IN_FP32) ? HIMUON_FP32 : HIMUON_BF16);
    if (st.enabled) per += ((d.flags & F_M_BF16) ? 2 : 4) + ((d.flags & F_OUT_FP32) ? 4 : 2);
    tile_bytes[i] = std::min<int64_t>(T, d.H) * std::min<int64_t>(T, d.W) * per;
  }

  const bool fp32 = p.path == HIMUON_PATH_FP32;
  // tensor path: T <= 32 one tile per warp (ns_mma32.cu); T = 64 and 128 on
  // one SM (ns_tc.cu); 128 < T <= 256 on a pair of SMs (ns_pair.cu); every
  // other T > 64, and the full-matrix map, as batched GEMMs (ns_gemm.cu)
  const bool warp_tiles = T <= 32;
  const bool onchip = T == 64 || T == 128;
  // 128 < T <= 256: one tile on a pair of SMs (ns_pair.cu); K = 0 has no
  // products and takes the GEMM path's gather/emit kernels
  const bool pair = T > 128 && T <= 256 && K > 0;
  if (!fp32 && !onchip && !warp_tiles && T < 64) {
    return fail(HIMUON_ERR_UNSUPPORTED,
                "tensor path: T = " + std::to_string(T) +
                    " is not implemented by this library; use T <= 32 or T >= 64, or the fp32 path");
  }

  // ---- TMA staging where the layouts allow it (16-byte aligned rows; for a
  // step bf16 G and fp32 M; T >= 64, since a 32-column box is narrower than the
  // 128-byte staging rows); other matrices are staged with plain loads. For a
  // step without weight decay, bf16 weights with 16-byte aligned rows are
  // updated by a TMA reduce-add (W += -lr s O) instead of a read-modify-write.
  std::vector<CUtensorMap> maps((fp32 || !onchip) ? 0 : 3 * static_cast<size_t>(n));
  for (int i = 0; i < n && !fp32 && onchip; ++i) {
    MatDesc& d = descs[i];
    const bool in32 = d.flags & F_IN_FP32;
    bool ok = (d.flags & F_IN_VEC) != 0 && T >= 64;
    if (st.enabled) ok = ok && !in32 && (d.flags & F_M_VEC) && !(d.flags & F_M_BF16);
    std::memset(&maps[3 * i], 0, 3 * sizeof(CUtensorMap));
    if (ok) ok = cached_map(h, &maps[3 * i], d.in, d.H, d.W, d.ld_in, in32, in32 ? 32 : 64, T);
    if (ok && st.enabled) ok = cached_map(h, &maps[3 * i + 1], d.mom, d.H, d.W, d.ld_mom, true, 32, T);
    if (ok) d.flags |= F_TMA;
    if (st.enabled && st.wd_factor == 1.f && !(d.flags & F_OUT_FP32) && (d.flags & F_OUT_VEC) &&
        cached_map(h, &maps[3 * i + 2], d.out, d.H, d.W, d.ld_out, false, 64, T))
      d.flags |= F_W_TMA;
  }

  // ---- per-matrix norm partials
  std::vector<int64_t> part_start(n + 1, 0);
  for (int i = 0; i < n; ++i) part_start[i + 1] = part_start[i] + cdiv(descs[i].H, NORM_ROWS_PER_PART);
  const int64_t nparts = (p.norm == HIMUON_NORM_MATRIX) ? part_start[n] : 0;

  // ---- workspace: [descs | part_start | tensor maps | partials]
  const size_t off_desc = 0;
  const size_t off_part = (sizeof(MatDesc) * n + 255) & ~size_t(255);
  const size_t off_maps = (off_part + sizeof(int64_t) * (n + 1) + 255) & ~size_t(255);
  const size_t off_partials = (off_maps + sizeof(CUtensorMap) * maps.size() + 255) & ~size_t(255);
  const size_t ws_need = off_partials + sizeof(float) * std::max<int64_t>(nparts, 1);
  const void* ws_before = h->ws;
  himuon_status s = grow(&h->ws, &h->ws_bytes, ws_need, stream, "workspace");
  if (s != HIMUON_OK) {
    h->ws_image.clear();
    return s;
  }
  if (h->ws != ws_before) h->ws_image.clear();
  h->host.assign(off_partials, 0);
  std::memcpy(h->host.data() + off_desc, descs.data(), sizeof(MatDesc) * n);
  std::memcpy(h->host.data() + off_part, part_start.data(), sizeof(int64_t) * (n + 1));
  if (!maps.empty())
    std::memcpy(h->host.data() + off_maps, maps.data(), sizeof(CUtensorMap) * maps.size());
  unsigned char* ws = static_cast<unsigned char*>(h->ws);
  // Pageable source: the copy is staged before cudaMemcpyAsync returns, so the
  // host buffer may be reused by the next call right away.
  cudaError_t e = cudaSuccess;
  if (h->ws_image != h->host) {
    e = cudaMemcpyAsync(ws, h->host.data(), off_partials, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) {
      h->ws_image.clear();
      return cuda_fail(e, "descriptor upload");
    }
    h->ws_image = h->host;
  }
  MatDesc* d_descs = reinterpret_cast<MatDesc*>(ws + off_desc);
  const int64_t* d_part = reinterpret_cast<const int64_t*>(ws + off_part);
  const void* d_maps = ws + off_maps;
  float* d_partials = reinterpret_cast<float*>(ws + off_partials);

  NSArgs ns;
  if ((s = make_ns_args(p, K, T, &ns)) != HIMUON_OK) return s;
  if (p.norm == HIMUON_NORM_MATRIX) {
    e = launch_matrix_norms(d_descs, n, d_part, nparts, d_partials, p.eps, st, stream);
    if (e != cudaSuccess) return cuda_fail(e, "matrix norm launch");
    h->launches += 2;
  }

  // ---- chunks: consecutive tile ranges whose input bytes stay within budget
  std::vector<std::pair<int64_t, int64_t>> chunks;
  if (chunk_bytes == 0) {
    chunks.emplace_back(0, total);
  } else {
    int64_t begin = 0, used = 0;
    for (int i = 0; i < n; ++i) {
      int64_t left = descs[i].ntiles, pos = descs[i].tile_start;
      const int64_t b = tile_bytes[i];
      while (left > 0) {
        const int64_t cap = static_cast<int64_t>(chunk_bytes) - used;
        int64_t k = std::min<int64_t>(left, cap >= b ? cap / b : 0);
        if (k == 0) {
          if (pos > begin) {                      // close the current chunk
            chunks.emplace_back(begin, pos);
            begin = pos;
            used = 0;
            continue;
          }
          k = 1;                                  // one tile above the budget
        }
        pos += k;
        left -= k;
        used += k * b;
      }
    }
    if (total > begin) chunks.emplace_back(begin, total);
  }

  if (fp32) {
    const int P = static_cast<int>(std::min<int64_t>(T, maxside));
    const size_t per_tile = size_t(3) * P * P * sizeof(float);
    int64_t nb = std::max<int64_t>(1, static_cast<int64_t>(kFp32ScratchCap / per_tile));
    nb = std::min<int64_t>(nb, 65535);
    int64_t biggest = 0;
    for (auto& c : chunks) biggest = std::max(biggest, c.second - c.first);
    nb = std::min(nb, biggest);
    void* scr = h->scratch;
    s = grow(&scr, &h->scratch_bytes, per_tile * nb, stream, "fp32 scratch");
    h->scratch = static_cast<float*>(scr);
    if (s != HIMUON_OK) return s;
    for (auto& c : chunks) {
      e = launch_ns_fp32(d_descs, n, c.first, c.second, T, P, ns, st, h->scratch, nb, stream);
      if (e != cudaSuccess) return cuda_fail(e, "fp32 path launch");
      const int64_t subs = (c.second - c.first + nb - 1) / nb;
      h->launches += subs * (2 + (ns.norm != HIMUON_NORM_NONE ? 1 : 0) + 3 * K);
    }
    return HIMUON_OK;
  }

  if (warp_tiles) {
    for (auto& c : chunks) {
      e = launch_ns_mma32(d_descs, n, c.first, c.second, ns, st, h->num_sms, stream);
      if (e != cudaSuccess) return cuda_fail(e, "tensor path launch");
      h->launches += 1;
    }
    return HIMUON_OK;
  }
  if (onchip) {
    for (auto& c : chunks) {
      e = launch_ns_tc(d_descs, d_maps, n, c.first, c.second, ns, st, h->wait_ns, h->d_err,
                       h->num_sms, stream);
      if (e != cudaSuccess) return cuda_fail(e, "tensor path launch");
      h->launches += 1;
    }
    return HIMUON_OK;
  }
  if (pair) {
    for (auto& c : chunks) {
      e = launch_ns_pair(d_descs, n, c.first, c.second, ns, st, h->wait_ns, h->d_err, h->num_sms,
                         stream);
      if (e != cudaSuccess) return cuda_fail(e, "tensor path launch");
      h->launches += 1;
    }
    return HIMUON_OK;
  }
  return run_gemm_path(h, descs, d_descs, T, ns, st, chunks, stream);
}

// Under HIMUON_PATH_AUTO, matrices this small or thin, and tiles of fewer than
// 64 elements, run on the fp32 path: with so few elements per tile the bf16
// rounding of the tensor path does not average out (errors of several percent
// on rank-1 matrices of a few elements, about 2 % on 1 x 1 tiles), and a
// tensor-core product would be almost all padding anyway.
bool needs_fp32(const MatDesc& d, int32_t T) {
  const int64_t th = std::min<int64_t>(T, d.H), tw = std::min<int64_t>(T, d.W);
  return std::min(d.H, d.W) <= 2 || static_cast<int64_t>(d.H) * d.W < 4096 || th * tw < 64;
}

// Runs the plan, with the small matrices of an AUTO-path request split off to
// the fp32 path (two plans on the same stream, so they run one after another).
himuon_status run_auto(himuon_handle* h, std::vector<MatDesc>& descs, int32_t T, int32_t K,
                       const himuon_ns_params& p, const StepArgs& st, size_t chunk_bytes,
                       cudaStream_t stream) {
  if (p.path != HIMUON_PATH_AUTO) return run_plan(h, descs, T, K, p, st, chunk_bytes, stream);
  std::vector<MatDesc> big, small;
  for (const MatDesc& d : descs) (needs_fp32(d, T) ? small : big).push_back(d);
  if (!big.empty()) {
    himuon_status s = run_plan(h, big, T, K, p, st, chunk_bytes, stream);
    if (s != HIMUON_OK) return s;
  }
  if (!small.empty()) {
    himuon_ns_params q = p;
    q.path = HIMUON_PATH_FP32;
    return run_plan(h, small, T, K, q, st, chunk_bytes, stream);
  }
  return HIMUON_OK;
}

int32_t in_flags(int32_t gtype, const void* g, int64_t ldg) {
  int32_t f = 0;
  if (gtype == HIMUON_FP32) f |= F_IN_FP32;
  if (aligned16(g, ldg, gtype)) f |= F_IN_VEC;
  return f;
}

}  // namespace

extern "C" {

int64_t himuon_launch_count(const himuon_handle* h) { return h ? h->launches : 0; }

int32_t himuon_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* himuon_last_error_string(void) { return g_last_error.c_str(); }

void himuon_default_ns_params(himuon_ns_params* p) {
  if (!p) return;
  p->a = 3.4445f;
  p->b = -4.7750f;
  p->c = 2.0315f;
  p->norm = HIMUON_NORM_TILE;
  p->eps = 1e-7f;
  p->path = HIMUON_PATH_AUTO;
  p->step_coeffs = nullptr;
}

double himuon_ns_flops(int64_t H, int64_t W, int32_t T, int32_t K) {
  if (H < 0 || W < 0 || T < 0 || K < 0) return 0.0;
  return 6.0 * static_cast<double>(H) * static_cast<double>(W) * static_cast<double>(T) *
         static_cast<double>(K);
}

int32_t himuon_schedule_tile(const int64_t* start_step, const int32_t* tile, int32_t n_points,
                             int64_t step) {
  if (!start_step || !tile || n_points < 1) return 0;
  for (int32_t i = 1; i < n_points; ++i)
    if (start_step[i] <= start_step[i - 1]) return 0;
  int32_t t = tile[0];
  for (int32_t i = 0; i < n_points; ++i)
    if (start_step[i] <= step) t = tile[i];
  return t;
}

himuon_status himuon_create(himuon_handle** out_handle) {
  if (!out_handle) return fail(HIMUON_ERR_INVALID_ARG, "out_handle is NULL");
  *out_handle = nullptr;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(HIMUON_ERR_NO_DEVICE, std::string("no CUDA device: ") + cudaGetErrorString(e));
  }
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(HIMUON_ERR_NO_DEVICE, "libhimuon is built for sm_103a (B300); device is sm_" +
                                          std::to_string(prop.major) + std::to_string(prop.minor));
  himuon_handle* h = new himuon_handle();
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  e = cudaMalloc(&h->d_err, 256);
  if (e == cudaSuccess) e = cudaMemset(h->d_err, 0, 256);
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "error word allocation");
  }
  *out_handle = h;
  return HIMUON_OK;
}

himuon_status himuon_destroy(himuon_handle* h) {
  if (!h) return HIMUON_OK;
  cudaDeviceSynchronize();
  if (h->ws) cudaFree(h->ws);
  if (h->scratch) cudaFree(h->scratch);
  if (h->tiles) cudaFree(h->tiles);
  if (h->d_err) cudaFree(h->d_err);
  delete h;
  return HIMUON_OK;
}

himuon_status himuon_set_wait_limit(himuon_handle* h, uint64_t ns) {
  if (!h) return fail(HIMUON_ERR_INVALID_ARG, "handle is NULL");
  if (ns == 0) return fail(HIMUON_ERR_INVALID_ARG, "wait limit must be > 0");
  h->wait_ns = ns;
  return HIMUON_OK;
}

himuon_status himuon_device_error(himuon_handle* h, void* stream, int32_t* code) {
  himuon_status s = check_handle(h);
  if (s != HIMUON_OK) return s;
  if (!code) return fail(HIMUON_ERR_INVALID_ARG, "code is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "stream sync");
  int v = 0;
  e = cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "error word read");
  e = cudaMemset(h->d_err, 0, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "error word clear");
  *code = v;
  return HIMUON_OK;
}

himuon_status himuon_wait_selftest(himuon_handle* h, void* stream) {
  himuon_status s = check_handle(h);
  if (s != HIMUON_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_wait_selftest(h->wait_ns, h->d_err, st);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test sync");
  return HIMUON_OK;
}

himuon_status himuon_tiled_ns(himuon_handle* h, const void* G, int64_t H, int64_t W, int64_t ldg,
                              int32_t gtype, int32_t T, int32_t K, const himuon_ns_params* params,
                              void* out, int64_t ldo, int32_t otype, void* stream) {
  himuon_matrix m;
  m.g = G;
  m.out = out;
  m.H = H;
  m.W = W;
  m.ldg = ldg;
  m.ldo = ldo;
  m.gtype = gtype;
  m.otype = otype;
  return himuon_tiled_ns_batched(h, &m, 1, T, K, params, 0, stream);
}

himuon_status himuon_tiled_ns_batched(himuon_handle* h, const himuon_matrix* mats, int32_t n,
                                      int32_t T, int32_t K, const himuon_ns_params* params,
                                      size_t chunk_bytes, void* stream) {
  himuon_status s = check_handle(h);
  if (s != HIMUON_OK) return s;
  if (!mats || n < 1) return fail(HIMUON_ERR_INVALID_ARG, "need at least one matrix");
  himuon_ns_params p;
  himuon_default_ns_params(&p);
  if (params) p = *params;
  if ((s = check_ns_params(p)) != HIMUON_OK) return s;
  if (T < 1) return fail(HIMUON_ERR_INVALID_ARG, "T must be >= 1");
  if (K < 0 || K > kMaxK) return fail(HIMUON_ERR_INVALID_ARG, "K must be in [0, 64]");
  {
    NSArgs probe;   // every step's coefficients checked before anything is enqueued
    if ((s = make_ns_args(p, K, T, &probe)) != HIMUON_OK) return s;
  }
  std::vector<MatDesc> descs(n);
  for (int32_t i = 0; i < n; ++i) {
    const himuon_matrix& m = mats[i];
    const std::string tag = "matrix " + std::to_string(i);
    if (!m.g || !m.out) return fail(HIMUON_ERR_INVALID_ARG, tag + ": NULL pointer");
    if (!valid_dtype(m.gtype) || !valid_dtype(m.otype))
      return fail(HIMUON_ERR_INVALID_ARG, tag + ": unknown dtype");
    if ((s = check_shape(m.H, m.W, m.ldg, (tag + " input").c_str())) != HIMUON_OK) return s;
    if ((s = check_shape(m.H, m.W, m.ldo, (tag + " output").c_str())) != HIMUON_OK) return s;
    if (m.g != m.out && overlaps(m.g, m.H, m.W, m.ldg, m.gtype, m.out, m.ldo, m.otype))
      return fail(HIMUON_ERR_INVALID_ARG, tag + ": output partially overlaps the input");
    if (m.g == m.out && (m.ldg != m.ldo || m.gtype != m.otype))
      return fail(HIMUON_ERR_INVALID_ARG, tag + ": in-place needs the same ld and dtype");
    MatDesc d{};
    d.in = m.g;
    d.out = m.out;
    d.mom = nullptr;
    d.ld_in = m.ldg;
    d.ld_out = m.ldo;
    d.ld_mom = 0;
    d.H = static_cast<int32_t>(m.H);
    d.W = static_cast<int32_t>(m.W);
    d.flags = in_flags(m.gtype, m.g, m.ldg);
    if (m.otype == HIMUON_FP32) d.flags |= F_OUT_FP32;
    if (aligned16(m.out, m.ldo, m.otype)) d.flags |= F_OUT_VEC;
    d.upd_scale = 0.f;
    d.norm_scale = 1.f;
    descs[i] = d;
  }
  StepArgs st{0.f, 1.f, 0, 0};
  return run_auto(h, descs, T, K, p, st, chunk_bytes, static_cast<cudaStream_t>(stream));
}

himuon_status himuon_step(himuon_handle* h, const himuon_param* params, int32_t n, int32_t T,
                          int32_t K, const himuon_ns_params* nsp, const himuon_step_params* step,
                          size_t chunk_bytes, void* stream) {
  himuon_status s = check_handle(h);
  if (s != HIMUON_OK) return s;
  if (!params || n < 1) return fail(HIMUON_ERR_INVALID_ARG, "need at least one parameter matrix");
  if (!step) return fail(HIMUON_ERR_INVALID_ARG, "step params are NULL");
  himuon_ns_params p;
  himuon_default_ns_params(&p);
  if (nsp) p = *nsp;
  if ((s = check_ns_params(p)) != HIMUON_OK) return s;
  if (T < 1) return fail(HIMUON_ERR_INVALID_ARG, "T must be >= 1");
  if (K < 0 || K > kMaxK) return fail(HIMUON_ERR_INVALID_ARG, "K must be in [0, 64]");
  {
    NSArgs probe;   // every step's coefficients checked before anything is enqueued
    if ((s = make_ns_args(p, K, T, &probe)) != HIMUON_OK) return s;
  }
  if (!std::isfinite(step->lr) || !std::isfinite(step->mu) || !std::isfinite(step->weight_decay))
    return fail(HIMUON_ERR_INVALID_ARG, "step params must be finite");
  if (!(step->scale_mode == 0 || step->scale_mode == 1))
    return fail(HIMUON_ERR_INVALID_ARG, "unknown scale mode");
  std::vector<MatDesc> descs(n);
  for (int32_t i = 0; i < n; ++i) {
    const himuon_param& q = params[i];
    const std::string tag = "param " + std::to_string(i);
    if (!q.w || !q.g || !q.m) return fail(HIMUON_ERR_INVALID_ARG, tag + ": NULL pointer");
    if (!valid_dtype(q.wtype) || !valid_dtype(q.gtype) || !valid_dtype(q.mtype))
      return fail(HIMUON_ERR_INVALID_ARG, tag + ": unknown dtype");
    if ((s = check_shape(q.H, q.W, q.ldw, (tag + " W").c_str())) != HIMUON_OK) return s;
    if ((s = check_shape(q.H, q.W, q.ldg, (tag + " G").c_str())) != HIMUON_OK) return s;
    if ((s = check_shape(q.H, q.W, q.ldm, (tag + " M").c_str())) != HIMUON_OK) return s;
    if (overlaps(q.w, q.H, q.W, q.ldw, q.wtype, q.g, q.ldg, q.gtype) ||
        overlaps(q.w, q.H, q.W, q.ldw, q.wtype, q.m, q.ldm, q.mtype) ||
        overlaps(q.g, q.H, q.W, q.ldg, q.gtype, q.m, q.ldm, q.mtype))
      return fail(HIMUON_ERR_INVALID_ARG, tag + ": W, G and M must not overlap");
    MatDesc d{};
    d.in = q.g;
    d.out = q.w;
    d.mom = q.m;
    d.ld_in = q.ldg;
    d.ld_out = q.ldw;
    d.ld_mom = q.ldm;
    d.H = static_cast<int32_t>(q.H);
    d.W = static_cast<int32_t>(q.W);
    d.flags = in_flags(q.gtype, q.g, q.ldg);
    if (q.wtype == HIMUON_FP32) d.flags |= F_OUT_FP32;
    if (aligned16(q.w, q.ldw, q.wtype)) d.flags |= F_OUT_VEC;
    if (q.mtype == HIMUON_BF16) d.flags |= F_M_BF16;
    if (aligned16(q.m, q.ldm, q.mtype)) d.flags |= F_M_VEC;
    const double sc = step->scale_mode == 0
                          ? std::sqrt(std::max(1.0, static_cast<double>(q.H) / static_cast<double>(q.W)))
                          : 1.0;
    d.upd_scale = static_cast<float>(static_cast<double>(step->lr) * sc);
    d.norm_scale = 1.f;
    descs[i] = d;
  }
  StepArgs st;
  st.mu = step->mu;
  st.wd_factor = static_cast<float>(1.0 - static_cast<double>(step->lr) * step->weight_decay);
  st.nesterov = step->nesterov ? 1 : 0;
  st.enabled = 1;
  return run_auto(h, descs, T, K, p, st, chunk_bytes, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
