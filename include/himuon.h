/*
 * himuon.h -- C ABI of the HiMuon tiled Newton-Schulz library (libhimuon.so).
 *
 * Method: "Hierarchical Muon: Tiled Newton-Schulz Updates for Efficient Muon
 * Optimization" (abstract). Muon-type optimizers turn a momentum-gradient matrix
 * into an update direction with a finite Newton-Schulz (NS) map (abstract,
 * sentence 1). HiMuon cuts each H x W matrix into T x T tiles, runs the same
 * finite NS map on every tile independently and reassembles the results
 * (sentence 3); for fixed T the work is O(H W T K) and splits into independent
 * small dense products (sentence 5), which is what enables tile-size-specific GPU
 * kernels, cross-layer batching, memory-bounded chunking and runtime tile-size
 * schedules (sentence 6).
 *
 * What this library computes (the abstract fixes the structure; the rest are
 * explicit parameters with the defaults below):
 *
 *   for every tile X (h x w, h = min(T, H - iT), w = min(T, W - jT)):
 *     X <- X * s           s = 1 / (||X||_F + eps)      (norm = TILE, default)
 *                          s = 1 / (||G||_F + eps)      (norm = MATRIX)
 *                          s = 1                        (norm = NONE)
 *     for k = 0 .. K-1:  A = X X^T;  B = b_k A + c_k A^2;  X <- a_k X + B X
 *     write X back at the tile's place.
 *   Defaults: (a_k, b_k, c_k) = (3.4445, -4.7750, 2.0315) for every k,
 *   eps = 1e-7.
 *
 * Conventions shared by every call below:
 *  - Matrices are row-major with a leading dimension (elements between the
 *    starts of consecutive rows), ld >= W. Pointers are DEVICE pointers, owned
 *    by the caller; the library never frees or keeps them past the call.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream). Errors found on the host are returned
 *    synchronously; the device error word (himuon_device_error) reports a wait
 *    that ran out of time inside a kernel.
 *  - `out` may be the same buffer as `G` (tiles are disjoint and each tile is
 *    read completely before it is written). Partial overlap is not allowed.
 *  - K = 0 is allowed: the output is the normalised input (NORM_NONE: a copy).
 *  - A handle owns a small device workspace (descriptor tables, per-matrix
 *    norms, scratch of the fp32 and large-tile paths). Calls that share a handle
 *    must be issued on one stream, or serialised by the caller.
 *  - Thread safety: handles are independent; the last-error string is per host
 *    thread.
 */
#ifndef HIMUON_H
#define HIMUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HIMUON_OK = 0,
  HIMUON_ERR_INVALID_ARG = 1,   /* bad size, pointer, ld, T, K or enum value */
  HIMUON_ERR_UNSUPPORTED = 2,   /* valid request this library does not implement */
  HIMUON_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  HIMUON_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out */
  HIMUON_ERR_NO_DEVICE = 5,     /* no usable sm_103 device */
  HIMUON_ERR_OUT_OF_MEMORY = 6  /* workspace could not be allocated */
} himuon_status;

typedef enum { HIMUON_BF16 = 0, HIMUON_FP32 = 1 } himuon_dtype;

typedef enum {
  HIMUON_NORM_TILE = 0,    /* per-tile Frobenius normalisation (default) */
  HIMUON_NORM_MATRIX = 1,  /* one factor from the whole matrix's Frobenius norm */
  HIMUON_NORM_NONE = 2     /* no normalisation */
} himuon_norm;

typedef enum {
  HIMUON_PATH_AUTO = 0,    /* bf16 tensor-core path; matrices with
                              min(H, W) <= 2 or fewer than 4096 elements, and
                              tiles of fewer than 64 elements (T < 8), run on
                              the fp32 path (too few elements for the bf16
                              rounding to average out) */
  HIMUON_PATH_TENSOR = 1,  /* same, requested explicitly */
  HIMUON_PATH_FP32 = 2     /* fp32 validation path (CUDA cores, fp32 FMA) */
} himuon_path;

/*
 * Parameters of the NS map. Fill with himuon_default_ns_params() first.
 *
 * Coefficients: by default every one of the K steps uses (a, b, c). A per-step
 * schedule (step_coeffs != NULL) gives step k its own (a_k, b_k, c_k): the
 * finite NS map is then the composition p_K o ... o p_1 of the odd polynomials
 * p_k(s) = a_k s + b_k s^3 + c_k s^5 on the singular values. A step with
 * c_k = 0 is a cubic step (two products instead of three), e.g. the classical
 * polar iteration (1.5, -0.5, 0). The abstract fixes neither the coefficients
 * nor that they are constant; both readings are parameters here. Every
 * coefficient must be finite, and a step with c_k != 0 must have |b_k / c_k|
 * and |e_k / c_k| <= 1e30, where e_k = a_k - min(a_k, 1.5) (HIMUON_ERR_INVALID_ARG
 * otherwise; the on-chip kernels start the A A accumulator at those ratios).
 */
typedef struct {
  float a, b, c;   /* NS coefficients of every step when step_coeffs is NULL */
  int32_t norm;    /* himuon_norm */
  float eps;       /* added to the Frobenius norm before dividing */
  int32_t path;    /* himuon_path */
  const float* step_coeffs;  /* NULL, or HOST memory with 3 * K floats
                                a_0, b_0, c_0, a_1, b_1, c_1, ...: the
                                coefficients of step k = 0 .. K-1 (read during
                                the call only; a, b, c are then ignored).
                                Non-finite values: HIMUON_ERR_INVALID_ARG. */
} himuon_ns_params;

/* One matrix of a cross-layer batch (himuon_tiled_ns_batched). */
typedef struct {
  const void* g;          /* input H x W, row-major, leading dimension ldg */
  void* out;              /* output H x W, leading dimension ldo; may equal g */
  int64_t H, W, ldg, ldo;
  int32_t gtype, otype;   /* himuon_dtype of g and out */
} himuon_matrix;

/* One weight matrix of a HiMuon step (himuon_step). */
typedef struct {
  void* w;                /* weights, updated in place */
  const void* g;          /* gradient */
  void* m;                /* momentum buffer, updated in place */
  int64_t H, W, ldw, ldg, ldm;
  int32_t wtype, gtype, mtype; /* himuon_dtype of w, g, m */
} himuon_param;

/* Optimizer parameters of a HiMuon step. */
typedef struct {
  float lr;             /* learning rate */
  float mu;             /* momentum coefficient */
  float weight_decay;   /* decoupled: W <- W - lr * weight_decay * W */
  int32_t nesterov;     /* 1: NS input U = G + mu * M_new; 0: U = M_new */
  int32_t scale_mode;   /* 0: s = sqrt(max(1, H / W)); 1: s = 1 */
} himuon_step_params;

/* Handle with its device workspace, bound to the current device at creation. */
typedef struct himuon_handle himuon_handle;

himuon_status himuon_create(himuon_handle** out_handle);
himuon_status himuon_destroy(himuon_handle* handle);

/* (a, b, c) = (3.4445, -4.7750, 2.0315), NORM_TILE, eps = 1e-7, PATH_AUTO,
   step_coeffs = NULL. */
void himuon_default_ns_params(himuon_ns_params* p);

/*
 * Tiled NS map of one matrix (abstract, sentences 3-5).
 * G: H x W input, ld ldg, dtype gtype (BF16 or FP32).
 * out: H x W output, ld ldo, dtype otype (BF16 or FP32); may be G itself.
 * T: tile size, 1 <= T. The tensor path keeps every tile on chip for all K
 *    steps for T <= 32 (one tile per warp, warp-level MMA), T = 64 and 128
 *    (one SM, tcgen05) and 128 < T <= 256 (one tile on a pair of SMs,
 *    tcgen05 cta_group::2); every other T >= 65 (and T >= max(H, W): one tile
 *    = the full-matrix map of Muon, sentences 1-2) runs as batched GEMMs;
 *    32 < T < 64 returns HIMUON_ERR_UNSUPPORTED there. The fp32 path takes any
 *    T.
 * K: number of NS steps, 0 <= K <= 64.
 * params: NULL means the defaults.
 * Returns HIMUON_ERR_INVALID_ARG for H or W < 1, ld < W, NULL pointers, bad
 * enums or T < 1, without touching the device.
 */
himuon_status himuon_tiled_ns(himuon_handle* handle, const void* G, int64_t H,
                              int64_t W, int64_t ldg, int32_t gtype, int32_t T,
                              int32_t K, const himuon_ns_params* params, void* out,
                              int64_t ldo, int32_t otype, void* stream);

/*
 * Cross-layer batch: the tiles of all n matrices form one work list that a
 * persistent kernel drains (abstract, sentence 6: cross-layer batching).
 * chunk_bytes: memory bound of one launch (abstract, sentence 6: memory-bounded
 * chunking). The work list is cut into chunks whose input tiles hold at most
 * chunk_bytes bytes (a chunk always holds at least one tile); each chunk is one
 * launch, and scratch of the scratch-using paths is sized by the chunk. 0 means
 * one chunk. The result does not depend on chunk_bytes.
 */
himuon_status himuon_tiled_ns_batched(himuon_handle* handle,
                                      const himuon_matrix* mats, int32_t n,
                                      int32_t T, int32_t K,
                                      const himuon_ns_params* params,
                                      size_t chunk_bytes, void* stream);

/*
 * One HiMuon optimizer step over n weight matrices, fused per tile:
 *   M <- mu M + G;  U = G + mu M (nesterov) or M;  O = tiled NS of U;
 *   W <- W - lr * weight_decay * W - lr * s * O,  s per matrix (scale_mode).
 * Momentum form, update scale and weight decay are not given by the abstract
 * (it only says the NS map acts on momentum-gradient matrices); they are the
 * explicit parameters above. W: BF16 or FP32; G: BF16 or FP32; M: FP32 or BF16.
 * T may change from call to call (runtime tile-size schedule, sentence 6).
 * W, G and M must not overlap one another.
 */
himuon_status himuon_step(himuon_handle* handle, const himuon_param* params,
                          int32_t n, int32_t T, int32_t K,
                          const himuon_ns_params* ns,
                          const himuon_step_params* step, size_t chunk_bytes,
                          void* stream);

/*
 * Runtime tile-size schedule helper (abstract, sentence 6). The schedule is
 * n_points pairs (start_step[i], T[i]) with increasing start_step; the T of the
 * last pair with start_step <= step is returned, T[0] before the first pair.
 * Returns 0 for an empty or unsorted schedule.
 */
int32_t himuon_schedule_tile(const int64_t* start_step, const int32_t* tile,
                             int32_t n_points, int64_t step);

/* Algorithmic flop count 6 * H * W * T * K of the tiled map (H, W, T, K >= 0). */
double himuon_ns_flops(int64_t H, int64_t W, int32_t T, int32_t K);

/*
 * Reads and clears the handle's device error word. Synchronises `stream`.
 * *code receives 0 (none) or a HIMUON_ERR_* value set by a kernel.
 */
himuon_status himuon_device_error(himuon_handle* handle, void* stream,
                                  int32_t* code);

/* Sets the limit of every bounded device-side wait (nanoseconds, > 0). */
himuon_status himuon_set_wait_limit(himuon_handle* handle, uint64_t ns);

/*
 * Self-test of the bounded wait: launches one kernel whose mbarrier wait can
 * never complete (nothing arrives), with the handle's wait limit. The kernel
 * gives up after the limit, records HIMUON_ERR_TIMEOUT in the device error word
 * and returns, so the context stays usable. Synchronises `stream`.
 */
himuon_status himuon_wait_selftest(himuon_handle* handle, void* stream);

/*
 * Size of the fixed device scratch of himuon_tiled_ns_fp32_noalloc (bytes).
 */
#define HIMUON_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/*
 * Allocation-free variant of the fp32 validation path of himuon_tiled_ns.
 * (The paper has no counterpart: this is a library convenience.)
 *
 * For callers that cannot call cudaMalloc: an application whose device memory
 * is all reserved by its own allocator (for example a framework's caching
 * allocator, or a process held to a fixed memory budget), or code that must
 * not block, since cudaMalloc/cudaFree can synchronise the device. Such
 * callers cannot create a handle, whose workspace is allocated on demand.
 * This call takes no handle and allocates nothing -- no cudaMalloc, no
 * cudaFree, no allocating library routine. Its scratch (the matrix descriptor,
 * per-matrix norm partials and the fp32 tile buffers) is one file-scope
 * device array of HIMUON_NOALLOC_SCRATCH_BYTES bytes, which every GPU that
 * loads the library holds until the process exits.
 *
 * Arguments, layout and result are those of himuon_tiled_ns with
 * params->path = HIMUON_PATH_FP32 (params->path is ignored here): G and out
 * are caller-owned device pointers, H x W row-major with leading dimensions
 * ldg / ldo; out may be G itself. The result equals that call's output.
 * Limit: one zero-padded tile of side P = min(T, max(H, W)) needs 12 * P * P
 * bytes (plus 4 bytes per 32 rows in NORM_MATRIX mode) and must fit in the
 * array, i.e. P <= 1182; larger requests return HIMUON_ERR_INVALID_ARG with a
 * message (himuon_last_error_string) naming the sizes, before any launch.
 * Larger tile counts are processed in sub-batches that fit.
 *
 * Set-up: the first call on a device (that device current) looks up the
 * array's device address with cudaGetSymbolAddress and caches it.
 * Concurrency: all calls share the one array, whose contents persist from
 * call to call (nothing in it needs clearing: each call writes every byte it
 * reads before reading it). Calls whose work overlaps on the GPU race on the
 * array and give wrong results: issue them on one stream. A call enqueues a
 * descriptor upload and then its kernels, so two host threads calling at the
 * same time can interleave those on one stream as well; a caller with several
 * host threads must serialise the calls itself, on the host.
 * Asynchronous on `stream` like the other calls.
 */
himuon_status himuon_tiled_ns_fp32_noalloc(const void* G, int64_t H, int64_t W,
                                           int64_t ldg, int32_t gtype, int32_t T,
                                           int32_t K, const himuon_ns_params* params,
                                           void* out, int64_t ldo, int32_t otype,
                                           void* stream);

/* Number of kernels this handle has launched so far (all calls, all paths). */
int64_t himuon_launch_count(const himuon_handle* handle);

/* Message of the last failing call on this host thread ("" if none). */
const char* himuon_last_error_string(void);

/* Version of the library as an integer (major * 10000 + minor * 100 + patch). */
int32_t himuon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HIMUON_H */
