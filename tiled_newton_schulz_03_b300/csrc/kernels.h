// Host-side launchers of the libhimuon kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <string>

#include "common.cuh"

namespace himuon {

// Tensor-core tiled NS, T in {64, 128} (ns_tc.cu). descs: device array of ndesc
// MatDesc; maps: device array of 2 * ndesc CUtensorMap (G, M), 64-byte aligned,
// valid for matrices flagged F_TMA; tiles [tile_begin, tile_end) of the flat
// tile list are processed. st.enabled selects the fused HiMuon step.
cudaError_t launch_ns_tc(const MatDesc* descs, const void* maps, int ndesc, int64_t tile_begin,
                         int64_t tile_end, const NSArgs& ns, const StepArgs& st, uint64_t wait_ns,
                         int* err, int num_sms, cudaStream_t stream);

// fp32 validation path (ns_fp32.cu): tiles (cut at multiples of T) padded to
// P x P (P = min(T, largest matrix side)) in a scratch buffer of 3 * nb * P * P
// floats; processes tiles [tile_begin, tile_end) in sub-batches of at most nb
// (<= 65535) tiles.
cudaError_t launch_ns_fp32(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                           int T, int P, const NSArgs& ns, const StepArgs& st, float* scratch,
                           int64_t nb, cudaStream_t stream);

// Per-matrix Frobenius norms (aux_kernels.cu): writes descs[m].norm_scale =
// 1 / (||X_m||_F + eps), where X is G (or the step's U). partials: device
// scratch of at least nparts_total floats; part_start: per-matrix offsets.
cudaError_t launch_matrix_norms(MatDesc* descs, int ndesc, const int64_t* part_start,
                                int64_t nparts_total, float* partials, float eps,
                                const StepArgs& st, cudaStream_t stream);
constexpr int NORM_ROWS_PER_PART = 32;

// One CTA waits on an mbarrier that nothing arrives on, for wait_ns, then
// records a time-out in *err and returns (aux_kernels.cu).
cudaError_t launch_wait_selftest(uint64_t wait_ns, int* err, cudaStream_t stream);

// Sets the message himuon_last_error_string() returns on this host thread (api.cu).
void record_last_error(const std::string& msg);

}  // namespace himuon
