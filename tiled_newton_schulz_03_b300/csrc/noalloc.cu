// Allocation-free entry point: the fp32 tiled NS map of one matrix with its
// scratch in a fixed, file-scope device array instead of a handle's workspace.
//
// Who needs it: callers that cannot call cudaMalloc at all -- an application
// whose device memory is entirely reserved by its own allocator (a framework's
// caching allocator that has already claimed the GPU, or a process held to a
// hard memory budget), or a loop that must never block, since cudaMalloc and
// cudaFree can synchronise the device. Such callers cannot create a
// himuon_handle (the handle allocates its workspace), so this entry point takes
// no handle and allocates nothing: the caller passes G and out, and everything
// else the fp32 path needs lives in g_noalloc_scratch below.
//
// The array costs kNoallocScratchBytes of device memory on every GPU that
// loads the library, held until the process exits.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/himuon.h"
#include "common.cuh"
#include "kernels.h"

using namespace himuon;

namespace {

constexpr size_t kNoallocScratchBytes = HIMUON_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
constexpr size_t kOffPart = 256;      // part_start[2]
constexpr size_t kOffPartials = 512;  // norm partials (matrix mode)

// Layout: [MatDesc | part_start[2] | per-matrix norm partials | fp32 tiles].
// Every byte a call reads is written earlier in the same call (descriptor and
// offsets by the upload, partials by the norm kernel, tiles by the gather
// kernel), so nothing has to be cleared between calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
bool g_scratch_ready[kMaxDevices] = {};

himuon_status nfail(himuon_status s, const std::string& msg) {
  record_last_error(msg);   // read back with himuon_last_error_string()
  return s;
}

int64_t esz(int32_t t) { return t == HIMUON_FP32 ? 4 : 2; }

bool vec_ok(const void* p, int64_t ld, int32_t t) {
  return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * esz(t)) % 16 == 0);
}

// Device address of g_noalloc_scratch on the current device. The host-side
// name of a __device__ array is only a stand-in, so the address is looked up
// once per device (with that device current) and cached.
himuon_status scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return nfail(HIMUON_ERR_NO_DEVICE, "device index out of range");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ready[dev]) {
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return nfail(HIMUON_ERR_CUDA, std::string("cudaGetDeviceProperties: ") + cudaGetErrorString(e));
    if (!(prop.major == 10 && prop.minor == 3))
      return nfail(HIMUON_ERR_NO_DEVICE, "libhimuon is built for sm_103a (B300)");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nfail(HIMUON_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ready[dev] = true;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return HIMUON_OK;
}

}  // namespace

extern "C" {

himuon_status himuon_tiled_ns_fp32_noalloc(const void* G, int64_t H, int64_t W, int64_t ldg,
                                           int32_t gtype, int32_t T, int32_t K,
                                           const himuon_ns_params* params, void* out, int64_t ldo,
                                           int32_t otype, void* stream) {
  // ---- arguments (same rules as himuon_tiled_ns)
  himuon_ns_params p;
  himuon_default_ns_params(&p);
  if (params) p = *params;
  if (!(p.norm == HIMUON_NORM_TILE || p.norm == HIMUON_NORM_MATRIX || p.norm == HIMUON_NORM_NONE))
    return nfail(HIMUON_ERR_INVALID_ARG, "ns params: unknown norm mode");
  if ((!p.step_coeffs && (!std::isfinite(p.a) || !std::isfinite(p.b) || !std::isfinite(p.c))) ||
      !std::isfinite(p.eps) || !(p.eps >= 0.f))
    return nfail(HIMUON_ERR_INVALID_ARG, "ns params: coefficients and eps must be finite, eps >= 0");
  if (!G || !out) return nfail(HIMUON_ERR_INVALID_ARG, "NULL pointer");
  if (!(gtype == HIMUON_BF16 || gtype == HIMUON_FP32) || !(otype == HIMUON_BF16 || otype == HIMUON_FP32))
    return nfail(HIMUON_ERR_INVALID_ARG, "unknown dtype");
  if (H < 1 || W < 1) return nfail(HIMUON_ERR_INVALID_ARG, "H and W must be >= 1");
  if (H > (1LL << 31) - 1024 || W > (1LL << 31) - 1024) return nfail(HIMUON_ERR_INVALID_ARG, "H or W too large");
  if (ldg < W || ldo < W) return nfail(HIMUON_ERR_INVALID_ARG, "leading dimension < W");
  if (T < 1) return nfail(HIMUON_ERR_INVALID_ARG, "T must be >= 1");
  if (K < 0 || K > 64) return nfail(HIMUON_ERR_INVALID_ARG, "K must be in [0, 64]");
  {
    const uintptr_t g0 = reinterpret_cast<uintptr_t>(G), o0 = reinterpret_cast<uintptr_t>(out);
    const uintptr_t g1 = g0 + static_cast<uintptr_t>(((H - 1) * ldg + W) * esz(gtype));
    const uintptr_t o1 = o0 + static_cast<uintptr_t>(((H - 1) * ldo + W) * esz(otype));
    if (G != out && g0 < o1 && o0 < g1)
      return nfail(HIMUON_ERR_INVALID_ARG, "output partially overlaps the input");
    if (G == out && (ldg != ldo || gtype != otype))
      return nfail(HIMUON_ERR_INVALID_ARG, "in-place needs the same ld and dtype");
  }

  // ---- coefficients of every step (checked before anything is enqueued)
  NSArgs ns;
  std::memset(&ns, 0, sizeof(ns));
  ns.eps = p.eps;
  ns.norm = p.norm;
  ns.K = K;
  ns.T = T;
  for (int32_t k = 0; k < K; ++k) {
    const float* c = p.step_coeffs ? p.step_coeffs + 3 * k : nullptr;
    ns.coef[k][0] = c ? c[0] : p.a;
    ns.coef[k][1] = c ? c[1] : p.b;
    ns.coef[k][2] = c ? c[2] : p.c;
    if (!std::isfinite(ns.coef[k][0]) || !std::isfinite(ns.coef[k][1]) || !std::isfinite(ns.coef[k][2]))
      return nfail(HIMUON_ERR_INVALID_ARG, "ns params: coefficients of step " + std::to_string(k) +
                                               " must be finite");
  }

  // ---- fit into the fixed scratch
  const int64_t P = std::min<int64_t>(T, std::max(H, W));
  const int64_t tiles_w = (W + T - 1) / T;
  const int64_t ntiles = ((H + T - 1) / T) * tiles_w;
  if (ntiles > (1LL << 31) - 1) return nfail(HIMUON_ERR_INVALID_ARG, "too many tiles");
  const int64_t nparts = (p.norm == HIMUON_NORM_MATRIX) ? (H + NORM_ROWS_PER_PART - 1) / NORM_ROWS_PER_PART : 0;
  const size_t off_tiles = kOffPartials + ((static_cast<size_t>(nparts) * sizeof(float) + 255) & ~size_t(255));
  const size_t per_tile = size_t(3) * static_cast<size_t>(P) * static_cast<size_t>(P) * sizeof(float);
  if (off_tiles + per_tile > kNoallocScratchBytes)
    return nfail(HIMUON_ERR_INVALID_ARG,
                 "request needs " + std::to_string(off_tiles + per_tile) + " bytes of scratch for one tile of " +
                     std::to_string(P) + " x " + std::to_string(P) + "; the fixed scratch holds " +
                     std::to_string(kNoallocScratchBytes) + " bytes (reduce T)");
  int64_t nb = static_cast<int64_t>((kNoallocScratchBytes - off_tiles) / per_tile);
  nb = std::min<int64_t>(std::min<int64_t>(nb, 65535), ntiles);

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return nfail(HIMUON_ERR_NO_DEVICE, std::string("no CUDA device: ") + cudaGetErrorString(e));
  }
  unsigned char* base = nullptr;
  himuon_status s = scratch_address(dev, &base);
  if (s != HIMUON_OK) return s;

  // ---- descriptor of the one matrix, uploaded into the scratch
  struct {
    MatDesc d;
    unsigned char pad[kOffPart - sizeof(MatDesc)];
    int64_t part_start[2];
  } host{};
  MatDesc& d = host.d;
  d.in = G;
  d.out = out;
  d.mom = nullptr;
  d.ld_in = ldg;
  d.ld_out = ldo;
  d.ld_mom = 0;
  d.H = static_cast<int32_t>(H);
  d.W = static_cast<int32_t>(W);
  d.tiles_w = static_cast<int32_t>(tiles_w);
  d.ntiles = static_cast<int32_t>(ntiles);
  d.tile_start = 0;
  d.flags = (gtype == HIMUON_FP32 ? F_IN_FP32 : 0) | (vec_ok(G, ldg, gtype) ? F_IN_VEC : 0) |
            (otype == HIMUON_FP32 ? F_OUT_FP32 : 0) | (vec_ok(out, ldo, otype) ? F_OUT_VEC : 0);
  d.upd_scale = 0.f;
  d.norm_scale = 1.f;
  host.part_start[0] = 0;
  host.part_start[1] = nparts;
  static_assert(sizeof(host) == kOffPart + 16, "upload layout");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Pageable source: staged before the call returns, so `host` may go out of scope.
  e = cudaMemcpyAsync(base, &host, sizeof(host), cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return nfail(HIMUON_ERR_CUDA, std::string("descriptor upload: ") + cudaGetErrorString(e));

  MatDesc* d_desc = reinterpret_cast<MatDesc*>(base);
  const int64_t* d_part = reinterpret_cast<const int64_t*>(base + kOffPart);
  float* d_partials = reinterpret_cast<float*>(base + kOffPartials);
  float* d_tiles = reinterpret_cast<float*>(base + off_tiles);

  StepArgs stp{0.f, 1.f, 0, 0};
  if (p.norm == HIMUON_NORM_MATRIX) {
    e = launch_matrix_norms(d_desc, 1, d_part, nparts, d_partials, p.eps, stp, st);
    if (e != cudaSuccess) return nfail(HIMUON_ERR_CUDA, std::string("matrix norm launch: ") + cudaGetErrorString(e));
  }
  e = launch_ns_fp32(d_desc, 1, 0, ntiles, T, static_cast<int>(P), ns, stp, d_tiles, nb, st);
  if (e != cudaSuccess) return nfail(HIMUON_ERR_CUDA, std::string("fp32 path launch: ") + cudaGetErrorString(e));
  return HIMUON_OK;
}

}  // extern "C"
