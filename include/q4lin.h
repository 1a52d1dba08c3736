/*
 * q4lin -- weight-only 4-bit linear layer  Y[N,T] = W[N,K] . X[K,T]  on GB300.
 *
 * Operation (the problem statement of the Q4 linear measurement report,
 * q4-linear.md, header table, and the linear-benchmark contract,
 * linear-benchmark.md, "status and scope" and section 4):
 *
 *   y[t*N + n] = bf16( sum_{k<K} w[n,k] * x[t*K + k] ),  accumulated in FP32,
 *   w[n,k]     = (q[n,k] - 8) * s[n*(Kp/64) + k/64],
 *   q[n,2j]    = wq[n*(Kp/2) + j] & 0xF,   q[n,2j+1] = wq[n*(Kp/2) + j] >> 4,
 *   Kp         = K rounded up to a multiple of 128 (K_pad).
 *
 * Weight format Q4_G64_FP16 "row-split" (linear-benchmark.md section 4,
 * format table: 32 code bytes + 2 scale bytes per group of 64; groups =
 * N * K_pad / 64): two separate planes, codes [N, Kp/2] uint8 and scales
 * [N, Kp/64] IEEE fp16, both row-major.  The plane positions k >= K are
 * padding: whatever bits they hold (NaN scale bits included) do not affect y.
 * X and Y are bf16, row-major [T, K] and [T, N] -- the same bytes as the
 * column-major X[K,T] / Y[N,T] views the report binds.  K must be a multiple
 * of 8, so that every X row starts 16-byte aligned.
 *
 * Ownership: the caller owns every buffer.  The library never allocates or
 * frees memory.  It keeps no state between calls except its error word and the
 * fixed scratch array of q4lin_linear_fp16_static (declared with it below).
 * Inputs (wq, scales, x, and LinearAdd's residual r unless it is y) are only
 * read.  Exactly the N*T elements of y are written.  The workspace belongs to
 * the call for its stream-ordered duration.
 *
 * Execution: every compute entry point is asynchronous on `stream` (a
 * cudaStream_t passed as void*; NULL = the legacy default stream), performs
 * no host synchronisation and no allocation, and may be captured into a CUDA
 * graph.  Results are deterministic run to run (no floating-point atomics).
 *
 * Errors: status codes (q4lin_status); no exception crosses this boundary.
 * Argument errors are detected on the host before anything is launched.
 * Device-side bounded waits that expire set a sticky device error word,
 * read with q4lin_device_status().
 */
#ifndef Q4LIN_H
#define Q4LIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  Q4LIN_OK = 0,
  Q4LIN_ERR_INVALID_ARG = 1,       /* null pointer with nonzero size, negative size, size overflow */
  Q4LIN_ERR_UNSUPPORTED_SHAPE = 2, /* K not a multiple of 8 */
  Q4LIN_ERR_MISALIGNED = 3,        /* a device pointer not 16-byte aligned */
  Q4LIN_ERR_WORKSPACE = 4,         /* workspace NULL while q4lin_workspace_bytes() > 0 */
  Q4LIN_ERR_DEVICE = 5,            /* current device is not compute capability 10.3 (the build targets sm_103a) */
  Q4LIN_ERR_CUDA = 6,              /* a CUDA runtime/driver call or a launch failed */
  Q4LIN_ERR_TIMEOUT = 7            /* a device-side bounded wait expired (see q4lin_device_status) */
} q4lin_status;

/* Routes: which kernel organisation q4lin_linear uses for a shape. */
typedef enum {
  Q4LIN_ROUTE_AUTO = 0,     /* let the library choose (what q4lin_linear does) */
  Q4LIN_ROUTE_GEMV = 1,     /* CUDA-core GEMV, weights decoded once per token block of <= 4 */
  Q4LIN_ROUTE_TC_SPLITK = 2,/* tcgen05 tile, K split across a thread-block cluster where the
                               planner finds it pays (what q4lin_linear uses from 33 tokens;
                               clusters up to 8, reducing through distributed shared memory
                               in rounds of as many partial tiles as the buffers hold) */
  Q4LIN_ROUTE_TC = 3,       /* tcgen05 tile, whole K per CTA */
  Q4LIN_ROUTE_TC_FP16 = 4,  /* opt-in: tcgen05 tile on fp16-rounded weights (see below) */
  Q4LIN_ROUTE_STREAM_MMA = 5/* streaming warp-MMA: weights streamed once by TMA, decoded in
                               registers to exact fp16 operands, reduced by mma.sync; X
                               converted by an operand pass (workspace); passes of 32 tokens */
} q4lin_route;

/*
 * Operand precision of the tile routes.  Q4LIN_ROUTE_TC and Q4LIN_ROUTE_TC_SPLITK
 * keep every product (q - 8) * x exact (bf16 operands) and apply the group scale
 * to FP32 per-group partial sums; they need no workspace.  The decode GEMV also
 * applies the scale in FP32.
 *
 * Q4LIN_ROUTE_TC_FP16 is never chosen by q4lin_linear.  It folds the scale into the
 * weight: each w = (q - 8) * s is rounded once to fp16 (taken at a power of two per
 * weight row so it cannot overflow), X is converted to fp16 exactly (taken at a
 * power of two per token), one FP32 tensor-memory accumulator sums the whole K
 * share, and the powers of two are undone on the FP32 result.  The weight rounding
 * (relative error at most 2^-11 per weight) puts rare outputs near y = 0 above the layer's
 * 1e-3 * rms(y) accuracy floor; its guaranteed bound is looser:
 * |y - y_ref| <= 8e-3 |y_ref| + 4e-3 rms(y_ref).  It needs workspace
 * (2*T*K + 4*T + 4*N bytes, each part rounded up to 256; q4lin_route_workspace_bytes)
 * and launches an operand pass before the tile kernel.
 */

/*
 * Bytes of device workspace q4lin_linear needs for (N, K, T); 0 means none
 * (the workspace pointer may then be NULL).  The linear-benchmark contract
 * (section 1.1) allocates workspace before timing through such a capacity
 * query.  Returns 0 for invalid sizes (q4lin_linear reports the error).
 * The value is a multiple of 256.
 */
size_t q4lin_workspace_bytes(int64_t N, int64_t K, int64_t T);

/*
 * Y = W . X (see the top of this file).
 *   wq        device, uint8  [N, Kp/2]  packed codes, 16-byte aligned
 *   scales    device, fp16   [N, Kp/64] bit patterns, 16-byte aligned
 *   x         device, bf16   [T, K]    bit patterns, 16-byte aligned
 *   y         device, bf16   [T, N]    bit patterns, 16-byte aligned (output)
 *   N, T      >= 0; N == 0 or T == 0 is an empty problem: Q4LIN_OK, nothing launched
 *   K         >= 0, multiple of 8; Kp = K rounded up to 128 (K == 0 writes y = +0)
 *   workspace device, >= q4lin_workspace_bytes(N, K, T) bytes, 256-byte aligned
 *   stream    cudaStream_t as void*
 * Returns Q4LIN_OK once the work is enqueued.
 */
int q4lin_linear(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y,
                 int64_t N, int64_t K, int64_t T, void* workspace, void* stream);

/*
 * Sibling weight formats of the format table (linear-benchmark.md section 4):
 * Q4G64_F16S (the layer's own), Q5G64_F16S (32 low + 8 high + 2 scale bytes
 * per 64 weights), Q6G64_F16S (32 + 16 + 2) and W8G32_F16S (32 code + 2 scale
 * bytes per 32 weights).  Readings (the table fixes only the byte counts):
 *   Q5 / Q6: codes = the Q4 code plane [N, Kp/2] (low 4 bits); high = [N, Kp/8]
 *     (Q5: bit b of byte i is bit 4 of weight 8i + b) or [N, Kp/4] (Q6: bits
 *     2b..2b+1 of byte i are bits 4..5 of weight 4i + b); w = (q - 16) * s,
 *     w = (q - 32) * s; scales [N, Kp/64].
 *   W8: codes [N, Kp] signed int8, w = code * s, scales [N, Kp/32].
 */
typedef enum {
  Q4LIN_QTYPE_Q4G64 = 0,
  Q4LIN_QTYPE_Q5G64 = 1,
  Q4LIN_QTYPE_Q6G64 = 2,
  Q4LIN_QTYPE_W8G32 = 3
} q4lin_qtype;

/*
 * Y = W . X for any of the formats above (arguments as q4lin_linear; `high`
 * is the Q5 / Q6 high-bit plane, 16-byte aligned, and is ignored otherwise).
 * Q4G64 is exactly q4lin_linear (workspace as q4lin_workspace_bytes).  The
 * other formats: Q5G64 and Q6G64 run on the decode GEMV for one token, on the
 * streaming warp-MMA route for 2..32 tokens (the high bits joined to the nibble
 * operands) and on the exact tile route beyond (token tiles up to 128 wide; the
 * high-bit plane is staged beside the codes); W8G32 runs on the decode GEMV for 1..4
 * tokens, on the warp-MMA route for 5..24 and on the exact tile route beyond (codes as
 * exact bf16, one accumulator per 32-wide scale group, token tiles up to 64 wide).  The
 * warp-MMA route's operand pass needs workspace: q4lin_qtype_workspace_bytes (256-byte
 * aligned, NULL allowed where that is 0).  Where a route has no shared-memory plan the
 * call falls back to another; shapes no route can plan return
 * Q4LIN_ERR_UNSUPPORTED_SHAPE.
 */
int q4lin_linear_qtype(int qtype, const uint8_t* codes, const uint8_t* high, const uint16_t* scales,
                       const uint16_t* x, uint16_t* y, int64_t N, int64_t K, int64_t T, void* workspace,
                       void* stream);

/* Workspace bytes q4lin_linear_qtype needs for this format and shape (0: none; a
 * multiple of 256; 0 for invalid sizes or an unknown format). */
size_t q4lin_qtype_workspace_bytes(int qtype, int64_t N, int64_t K, int64_t T);

/* The route q4lin_linear_qtype takes for this format and shape on the current device
 * (host-only logic; Q4LIN_ROUTE_GEMV also for shapes it refuses), -1 for an unknown
 * format or invalid sizes. */
int q4lin_qtype_route(int qtype, int64_t N, int64_t K, int64_t T);

/*
 * LinearAdd (a fused operation the linear-benchmark page names and leaves to its
 * own benchmark; the reading here): y = W . x + r, the bf16 residual r [T, N]
 * (row-major like y, 16-byte aligned) added to the FP32 sum before y's one bf16
 * rounding.  r may be y itself (in-place residual add); otherwise r and y must not
 * overlap.  No workspace: up to 8 tokens it runs the streaming warp-MMA route's
 * one-launch form (its kernel converts X into shared memory itself; the residual joins
 * the sum in the epilogue) where that form's shared-memory plan fits, otherwise the
 * exact tile route (q4lin_fused_route tells which).  Other arguments and errors as
 * q4lin_linear; r NULL gives Q4LIN_ERR_INVALID_ARG.  K = 0 gives y = r.
 */
int q4lin_linear_add(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, const uint16_t* r, uint16_t* y,
                     int64_t N, int64_t K, int64_t T, void* stream);

/*
 * LinearSwiGLU (a fused operation the linear-benchmark page names and leaves to its
 * own benchmark; the reading here): one packed weight of 2F rows -- rows [0, F) the
 * gate projection, rows [F, 2F) the up projection (the MLP gate/up parent of the
 * page's model suites, 34816 = 2 x 17408 rows) -- applied to x, and
 *   y[t*F + f] = bf16( silu(g) * u ),  g = (W x)[t, f],  u = (W x)[t, F + f],
 *   silu(z) = z / (1 + e^-z), all in FP32 before the one bf16 rounding.
 *   wq        device, uint8 [2F, Kp/2]; scales device, fp16 [2F, Kp/64]
 *   x         device, bf16 [T, K];     y device, bf16 [T, F] (output)
 * No workspace.  Up to 8 tokens, where its shared-memory plan fits, the streaming
 * warp-MMA route's one-launch form: each CTA streams a band of gate rows, then the band
 * of up rows that pairs with it, and forms the product at the up band's end.  Otherwise
 * the exact tile route: a tile stacks 64 gate rows over the matching 64 up rows, and the
 * product is formed in the epilogue.  Alignment, sizes and errors as q4lin_linear (with
 * N = 2F).  K = 0 gives y = +0.
 */
int q4lin_linear_swiglu(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y, int64_t F,
                        int64_t K, int64_t T, void* stream);

/*
 * LinearPair (a fused operation the linear-benchmark page names; the reading here):
 * two packed weights applied to the same x in one call, y_a = W_a x and y_b = W_b x.
 *   wq_a / scales_a  [N_a, Kp/2] / [N_a, Kp/64];  wq_b / scales_b  [N_b, Kp/2] / [N_b, Kp/64]
 *   x  bf16 [T, K];  y_a  bf16 [T, N_a];  y_b  bf16 [T, N_b] (outputs, must not overlap)
 * Up to 8 tokens, where the streaming warp-MMA route's one-launch form fits both
 * weights, one launch of it per weight; otherwise the exact tile route in one launch
 * (plus a tail launch where the planner splits the last wave): the row tiles of W_a are
 * followed by those of W_b, and both read the same X tiles.  No workspace.  Alignment
 * and errors as q4lin_linear; N_a or N_b may be 0 (that output is not touched).  K = 0
 * gives zeros.
 */
int q4lin_linear_pair(const uint8_t* wq_a, const uint16_t* scales_a, const uint8_t* wq_b, const uint16_t* scales_b,
                      const uint16_t* x, uint16_t* y_a, uint16_t* y_b, int64_t N_a, int64_t N_b, int64_t K, int64_t T,
                      void* stream);

/*
 * The route a fused operation takes for (N, K, T) on the current device (host-only
 * logic): op 1 LinearAdd (N rows), 2 LinearSwiGLU (N = F), 3 LinearPair (N = rows of
 * each weight).  Returns Q4LIN_ROUTE_STREAM_MMA (the one-launch warp-MMA form, one
 * launch per weight) or Q4LIN_ROUTE_TC_SPLITK, -1 for an unknown op or invalid sizes.
 */
int q4lin_fused_route(int op, int64_t N, int64_t K, int64_t T);

/*
 * Kernels one q4lin_linear_qtype call of this format and shape launches (0 for a
 * shape it refuses or an unknown format); Q4G64 is q4lin_kernel_launches.
 */
int q4lin_qtype_kernel_launches(int qtype, int64_t N, int64_t K, int64_t T);

/*
 * Diagnostic form of q4lin_linear that runs a given route instead of the
 * library's choice (the same arguments; route Q4LIN_ROUTE_AUTO is
 * q4lin_linear itself).  Tests use it to compare every route with the
 * oracle on the same shapes; the benchmark never does.  Workspace
 * requirement: q4lin_route_workspace_bytes(route, N, K, T).
 */
int q4lin_linear_route(int route, const uint8_t* wq, const uint16_t* scales, const uint16_t* x,
                       uint16_t* y, int64_t N, int64_t K, int64_t T, void* workspace, void* stream);

/*
 * The fp16 tile route (Q4LIN_ROUTE_TC_FP16, the same kernels and bound) for callers
 * that cannot allocate device memory: no workspace argument, and the call allocates
 * nothing.  The pages describe no such entry point; it exists for code that must
 * not call cudaMalloc around the layer (work issued inside a capture that may not
 * allocate, an allocator that owns the device, a host without an allocator).
 *   Scratch: a fixed 16 MiB device array inside the library, which every process
 *     that loads the library holds on each GPU it uses until it exits.  Shapes whose
 *     2*T*K + 4*T + 4*N bytes (each part rounded up to 256) exceed it return
 *     Q4LIN_ERR_UNSUPPORTED_SHAPE (N = 6144, K = 5120 fits up to T = 1635).
 *   Set-up: the first call in each CUDA context (per device, and again after a
 *     cudaDeviceReset) looks up the array's device address (one
 *     cudaGetSymbolAddress, no allocation); make that first call before any stream
 *     capture on that device.
 *   Sharing: every call uses the same array, so calls that overlap on the GPU (in
 *     different streams, or from different host threads) race on it; order them.
 *     Each call rewrites all the scratch it reads, so nothing needs clearing.
 * Arguments, alignment, ownership of inputs and outputs and the other error codes
 * are those of q4lin_linear.
 */
int q4lin_linear_fp16_static(const uint8_t* wq, const uint16_t* scales, const uint16_t* x, uint16_t* y,
                             int64_t N, int64_t K, int64_t T, void* stream);

/*
 * q4lin_linear with X and Y in page-locked host memory (cudaHostAlloc, or
 * cudaHostRegister'ed and mapped), for callers whose activations live on the host.
 * The pages describe no such entry point.  In stream order: a kernel copies X from
 * x_host into the workspace (SM loads of the page-locked memory, chained to the
 * layer by programmatic dependent launch), then q4lin_linear runs on it (its own
 * route choice) and its kernels store Y straight into y_host (every route writes Y
 * with plain stores; K == 0 stages the zeros in the workspace and copies them out).
 *   x_host     page-locked host, bf16 [T, K], 16-byte aligned (read only)
 *   y_host     page-locked host, bf16 [T, N], 16-byte aligned (fully overwritten
 *              once the stream reaches the end of the call)
 *   workspace  device, >= q4lin_host_workspace_bytes(N, K, T) bytes, 256-byte
 *              aligned: X staging (2TK bytes), Y staging (2TN bytes, used when
 *              K == 0), each rounded up to 256, then q4lin_linear's own workspace
 *   wq, scales, N, K, T, stream: as q4lin_linear.
 * A pointer that is not page-locked host memory of this process (pageable memory,
 * device memory) returns Q4LIN_ERR_INVALID_ARG with a detail, before any launch.
 * The host buffers belong to the call until the stream passes it: do not touch them
 * (or free them) before then.
 */
size_t q4lin_host_workspace_bytes(int64_t N, int64_t K, int64_t T);
int q4lin_linear_host(const uint8_t* wq, const uint16_t* scales, const uint16_t* x_host, uint16_t* y_host,
                      int64_t N, int64_t K, int64_t T, void* workspace, void* stream);
size_t q4lin_route_workspace_bytes(int route, int64_t N, int64_t K, int64_t T);

/* The route q4lin_linear picks for (N, K, T) on the current device (host-only logic). */
int q4lin_select_route(int64_t N, int64_t K, int64_t T);

/*
 * The tile plan a tensor-core route runs for (N, K, T) on the current device:
 *   *tile_n        token-tile width of one CTA (the MMA N: 16, 32, 64, 128 or 256)
 *   *split_k       CTAs of one thread-block cluster that share the K range of a
 *                  tile in the main launch
 *   *main_tiles    output tiles (128 rows x tile_n tokens, numbered with the row
 *                  tile fastest) covered by the main launch; may be NULL
 *   *tail_split_k  cluster size of a second launch over the remaining tiles
 *                  (whole waves run unsplit, the partial last wave split along
 *                  K), 0 when there is none; may be NULL
 * route Q4LIN_ROUTE_AUTO resolves as q4lin_linear does; the GEMV route (or an
 * empty problem) gives *tile_n = 0, *split_k = 1, *main_tiles = 0,
 * *tail_split_k = 0.  Host-only logic: reads device attributes and occupancy,
 * launches nothing.  Returns Q4LIN_OK, or Q4LIN_ERR_INVALID_ARG for NULL
 * tile_n / split_k, an unknown route or invalid sizes (outputs untouched).
 */
int q4lin_tile_plan(int route, int64_t N, int64_t K, int64_t T, int* tile_n, int* split_k, int64_t* main_tiles,
                    int* tail_split_k);

/* Number of kernel launches one q4lin_linear call issues for (N, K, T) (host-only logic; 0 for
 * an empty problem or invalid sizes). */
int q4lin_kernel_launches(int64_t N, int64_t K, int64_t T);

/* Human-readable text of a q4lin_status (never NULL). */
const char* q4lin_status_string(int status);

/*
 * Sticky device-side error word of the current device (0 = none; otherwise a
 * q4lin_status, e.g. Q4LIN_ERR_TIMEOUT, set by a kernel whose bounded wait
 * expired).  Synchronises the device to read it.  q4lin_clear_device_status
 * resets it to 0.  Both return Q4LIN_ERR_CUDA (as the value) if the read fails.
 */
int q4lin_device_status(void);
int q4lin_clear_device_status(void);

/* Text describing the last error a q4lin call returned on this host thread (which call failed
 * and the CUDA error text, if any); "" if the last call succeeded.  Owned by the library, valid
 * until the next q4lin call on the same thread. */
const char* q4lin_last_error_detail(void);

/*
 * Diagnostics (no counterpart in the layer's operation).
 *
 * HBM read probe: the pure-read ceiling the linear-benchmark contract (section 4,
 * theoretical traffic) prefers to a copy for a weight-streaming GEMV.  Reads
 * `bytes` bytes at `src` (device, 16-byte aligned; bytes a multiple of 16) with
 * 16-byte non-allocating loads in a grid-stride loop of `blocks` CTAs of 512
 * threads (blocks <= 0: four per SM), and writes one XOR word per CTA to `sink`
 * (device, >= blocks words) so the loads cannot be removed.  Asynchronous on
 * `stream`; the caller times it.  Returns Q4LIN_OK once enqueued,
 * Q4LIN_ERR_INVALID_ARG / Q4LIN_ERR_MISALIGNED for bad arguments.
 */
int q4lin_hbm_read_probe(const void* src, size_t bytes, uint32_t* sink, int blocks, void* stream);

/*
 * Wait-expiry check: one warp runs the kernels' bounded mbarrier wait, with the
 * bound `limit` polls (1 .. 2^20; each poll suspends for at most about a
 * microsecond), on a phase that nothing ever completes.  The wait must expire:
 * the kernel records Q4LIN_ERR_TIMEOUT in the device error word that
 * q4lin_device_status() reports, raises its CTA's abort flag and returns.  `out`
 * (device, one int) receives 1 if the wait succeeded (it cannot) plus 2 if the
 * abort flag was raised.  Asynchronous on `stream`.  It faults and hangs nothing;
 * it exists so that tests can check the timeout path on a live GPU.
 */
int q4lin_diag_wait_expiry(uint32_t limit, int* out, void* stream);

/* Library version, "major.minor.patch". */
const char* q4lin_version(void);

#ifdef __cplusplus
}
#endif

#endif /* Q4LIN_H */
