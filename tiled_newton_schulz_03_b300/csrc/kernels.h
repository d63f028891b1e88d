// Host-side launchers of the libhimuon kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <string>

#include "../../include/himuon.h"
#include "common.cuh"

namespace himuon {

// Tensor-core tiled NS, T in {64, 128} (ns_tc.cu). descs: device array of ndesc
// MatDesc; maps: device array of 3 * ndesc CUtensorMap (G, M, W), 64-byte
// aligned; G and M valid for matrices flagged F_TMA, W for those flagged
// F_W_TMA; tiles [tile_begin, tile_end) of the flat tile list are processed.
// st.enabled selects the fused HiMuon step.
cudaError_t launch_ns_tc(const MatDesc* descs, const void* maps, int ndesc, int64_t tile_begin,
                         int64_t tile_end, const NSArgs& ns, const StepArgs& st, uint64_t wait_ns,
                         int* err, int num_sms, cudaStream_t stream);

// Tensor-core tiled NS for 128 < T <= 256, K >= 1 (ns_pair.cu): one tile per
// cluster of two CTAs (cta_group::2 products), held on chip for all K steps;
// plain global loads and stores (any alignment). Same arguments as
// launch_ns_tc without the tensor maps.
cudaError_t launch_ns_pair(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                           const NSArgs& ns, const StepArgs& st, uint64_t wait_ns, int* err,
                           int num_sms, cudaStream_t stream);

// Tensor-core tiled NS for T <= 32 (ns_mma32.cu): one warp per tile, warp-level
// mma.sync; any alignment, plain loads. Same arguments as launch_ns_tc without
// the tensor maps and the wait limit (nothing waits on another thread).
cudaError_t launch_ns_mma32(const MatDesc* descs, int ndesc, int64_t tile_begin, int64_t tile_end,
                            const NSArgs& ns, const StepArgs& st, int num_sms, cudaStream_t stream);

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

// Batched-GEMM path for large tiles and the full-matrix map (ns_gemm.cu): n
// tiles of one padded oriented shape Hp x Wp (multiples of 128, Hp <= Wp),
// d_tiles their device descriptors, scratch of gemm_scratch_bytes(Hp, Wp) * n
// bytes. *status is set to a non-OK value if a tensor map cannot be encoded.
cudaError_t launch_ns_gemm_batch(const GTile* d_tiles, int n, int Hp, int Wp, const MatDesc* descs,
                                 const NSArgs& ns, const StepArgs& st, void* scratch,
                                 uint64_t wait_ns, int* err, cudaStream_t stream,
                                 himuon_status* status);
int64_t gemm_scratch_bytes(int Hp, int Wp);

// 3-D tiled bf16 tensor map over n row-major C x R matrices stored back to back,
// box of box_c columns x box_r rows x 1, 128-byte swizzle, zero fill (api.cu).
bool encode_map_3d(void* map, const void* base, int64_t C, int64_t R, int64_t n, int box_c,
                   int box_r);

// Sets the message himuon_last_error_string() returns on this host thread (api.cu).
void record_last_error(const std::string& msg);

}  // namespace himuon
