/*
 * gptq_fold.h -- C ABI of the GB300 GPTQ fold + q4tp / q2tp sweep library
 * (libgptqfold.so).
 *
 * What it computes is defined by two pages of the cortiq project:
 *   [fold page]  cortiq-engine src/gpu_wgpu/gptq_dev.rs -- module doc comment
 *                (steps 1-5), WGSL kernels build_a, chol_*, inv_*, make_u,
 *                q4tp_group, q4tp_trail, and the host functions fold /
 *                sweep_q4tp;
 *   [host page]  cortiq-cli src/gptq.rs -- gptq_fold_operator_par (the f64
 *                host fold), gptq_quantize_q4tp (host sweep) and
 *                gptq_quantize_q4tp_dev (ladder tables handed to the device).
 *
 * Conventions (all entry points):
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     the comment says "host".  The library never frees or keeps a caller
 *     buffer, and allocates no device memory itself: scratch comes from the
 *     caller's workspace (size from the matching *_workspace_bytes call).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Calls return once the work is enqueued, except gptq_fold and
 *     gptq_quantize_group, which read back one 4-byte pivot flag per
 *     factorisation attempt (a stream synchronisation) to decide the damping.
 *   - float buffers must be 16-byte aligned; shapes are checked before any
 *     launch.  Errors come back as a gptq_status; nothing traps.
 *   - Matrices are row-major and dense (leading dimension = column count).
 */
#ifndef GPTQ_FOLD_H
#define GPTQ_FOLD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GPTQ_OK = 0,
  GPTQ_ERR_ARG = 1,      /* null or misaligned pointer, lambda not finite  */
  GPTQ_ERR_SHAPE = 2,    /* n, rows out of range; n % 32 != 0 for a sweep  */
  GPTQ_ERR_NOMEM = 3,    /* workspace smaller than *_workspace_bytes       */
  GPTQ_ERR_NOT_SPD = 4,  /* damping raised past lambda = 10 still failed   */
  GPTQ_ERR_CUDA = 5,     /* a CUDA runtime call or launch failed           */
  GPTQ_ERR_TIMEOUT = 6   /* a bounded device-side wait gave up             */
} gptq_status;

/* Largest n / rows accepted (n * n floats must stay addressable by int64). */
#define GPTQ_MAX_N 65536
#define GPTQ_MAX_ROWS (1 << 24)
#define GPTQ_GROUP 32

/* Human-readable name of a status code (static string). */
const char* gptq_status_string(int status);

/* Workspace bytes gptq_fold needs for n channels (0 if n is out of range). */
size_t gptq_fold_workspace_bytes(int n);

/*
 * gptq_fold -- the fold operator of one Hessian group.
 * [fold page] module doc, steps 1-4; kernels diag_get, build_a, chol_diag,
 * chol_panel, chol_update, inv_diag, inv_rows, inv_update, make_u; host fn
 * fold / fold_inner (damping retry).
 *
 *   H_packed  in   f32, n(n+1)/2: upper triangle of H by rows (row r starts
 *                  at r(2n-r+1)/2, element (a<=b) at start(a)+(b-a)).  Not
 *                  modified.
 *   n         in   channels, 1 <= n <= GPTQ_MAX_N.
 *   lambda    in   relative damping (the pages use 0.01); negative -> 0.
 *   U         out  f32 n*n row-major: upper Cholesky factor of H_d^-1
 *                  (U^T U = H_d^-1, U_jj > 0, zeros below the diagonal),
 *                  H_d = H + lambda_used * max(mean(diag), 1e-12) * I with
 *                  dead channels (!(H_ii > 0)) replaced by a unit row/column.
 *   D         out  f32 n (may be NULL): sqrt(H_ii + damp) for a live channel,
 *                  -sqrt(1 + damp) for a dead one (sign marks dead).
 *   hdiag     out  f32 n (may be NULL): raw H_ii, the sweep's rung weights.
 *   lambda_used out host double (may be NULL): the damping that factored.
 *   ws, ws_bytes   workspace, >= gptq_fold_workspace_bytes(n), 256-B aligned.
 *
 * Damping retry (fold page, fold_inner): a pivot that is not positive (or
 * NaN) raises lambda (0 -> 1e-4, otherwise x10) and refactors from H; past
 * 10 the call returns GPTQ_ERR_NOT_SPD (U then holds no valid operator).
 */
gptq_status gptq_fold(const float* H_packed, int n, double lambda, float* U, float* D,
                      float* hdiag, double* lambda_used, void* ws, size_t ws_bytes,
                      void* stream);

/*
 * gptq_ladder -- per-row q4tp scale ladder (a7).  The pages only call the
 * converter that makes it (host page, gptq_quantize_q4tp_dev: "the
 * converter's ladder", rungs 2^(lo + c*step), f16 lo/step); the reading
 * implemented: over the row's groups with absmax a_g > 0, x_g = f32(a_g/7),
 * lo = f16(log2 min x_g), step = f16(max(0, (log2 max x_g - lo)/31)) (0 when
 * min == max), tab[c] = f32(2^(lo + c*step)); an all-zero row gets zeros.
 *
 *   W     in  f32 rows*n (dead columns already zeroed), n % 32 == 0.
 *   tab   out f32 rows*32;  lost out f32 rows*2 = (lo, step) per row.
 */
gptq_status gptq_ladder(const float* W, int rows, int n, float* tab, float* lost, void* stream);

/* Workspace bytes for gptq_q4tp_sweep / gptq_q2tp_sweep: residuals of four
 * 128-column blocks go into the later columns in one update (K = 512).  A
 * workspace of at least half that (rows*2048 + n*2048 bytes, plus slack)
 * is accepted and runs pairs of blocks (K = 256): the same mathematics, a
 * different f32 summation order in the updates. */
size_t gptq_sweep_workspace_bytes(int rows, int n);

/*
 * gptq_q4tp_sweep -- the column-sequential q4tp GPTQ sweep of W against U.
 * [fold page] module doc step 5, WGSL q4tp_group + q4tp_trail, host fn
 * sweep_q4tp; [host page] gptq_quantize_q4tp (same rule, host form).
 *
 * Per 32-column group: rung = best of nominal-2..nominal+1 by the
 * hw-weighted error (nominal from the corrected absmax), codes
 * clamp(rne(w/s), -8, 7), residual e_j = (w_j - q s)/U_jj with in-group
 * feedback; the residuals reach the later columns through
 * W[:, later] -= E * U[group, later] (applied here per block of 128 columns:
 * same mathematics, different f32 summation order than one group at a time).
 *
 *   W       in/out f32 rows*n: the weights (dead columns zeroed); consumed
 *                  (holds partially corrected values afterwards).
 *   U       in  f32 n*n from gptq_fold.   hw in f32 n: rung-error weights
 *                  (the pages pass the raw H_ii).
 *   tab, lost in  from gptq_ladder.
 *   nibbles out u8 rows*n/2: tile (row, group) = 16 bytes at
 *                  (row*n/32 + group)*16; column j -> byte j/2, low nibble
 *                  for even j; nibble = code + 8.
 *   rungs   out u8 rows*n/32 (rung index 0..31 per (row, group)).
 *   scales  out f32 rows*n/32 = tab[row][rung].
 *   n % 32 == 0 (else GPTQ_ERR_SHAPE, as the fold page's sweep declines).
 */
gptq_status gptq_q4tp_sweep(float* W, int rows, int n, const float* U, const float* hw,
                            const float* tab, const float* lost, uint8_t* nibbles,
                            uint8_t* rungs, float* scales, void* ws, size_t ws_bytes,
                            void* stream);

/*
 * gptq_q4tp_group -- the rung + rounding + in-group feedback rule alone, on
 * one 32-column tile of every row ([fold page] WGSL q4tp_group).  Exposed so
 * the rule can be checked bit for bit against a reference on given tiles.
 *
 *   tile  in  f32 rows*32 (the group's current weights per row).
 *   ublk  in  f32 32*32 row-major: U[c0..c0+32, c0..c0+32].
 *   hw    in  f32 32.  tab/lost in as for the sweep (rows*32, rows*2).
 *   nibbles out u8 rows*16; rungs out u8 rows; scales out f32 rows;
 *   E     out f32 rows*32 (the scaled residuals e_j).
 */
gptq_status gptq_q4tp_group(const float* tile, int rows, const float* ublk, const float* hw,
                            const float* tab, const float* lost, uint8_t* nibbles,
                            uint8_t* rungs, float* scales, float* E, void* stream);

/*
 * gptq_q4tp_sweep_noalloc -- gptq_q4tp_sweep for callers that cannot
 * allocate device memory and have no workspace to lend.  Two kinds of caller
 * are meant: a plugin or custom operator inside a host framework that owns
 * every device allocation (its pool or budget is not reachable from here) and
 * hands the plugin only the input and output buffers; and a latency-bound
 * caller that must keep cudaMalloc off its hot path, because cudaMalloc can
 * synchronise the whole device and stall the caller's other streams.  The
 * pages have no counterpart; it is a packaging of the same sweep.
 *
 * Arguments, layouts and results are those of gptq_q4tp_sweep, without
 * ws/ws_bytes.  Scratch lives instead in one file-scope device array of
 * GPTQ_SWEEP_NOALLOC_SCRATCH_BYTES per GPU, which every GPU that loads the
 * library holds until the process exits.  It fits shapes with
 * rows*2048 + n*2048 bytes (plus slack) <= that size (about rows + n <= 24575,
 * e.g. 5120 rows x 17408 channels); larger shapes return GPTQ_ERR_NOMEM
 * before any work.  Where the array also holds gptq_sweep_workspace_bytes
 * (about rows + n <= 12287) the result is the workspace call's bit for bit;
 * otherwise it runs pairs of blocks per update (same mathematics, different
 * f32 summation order), as gptq_q4tp_sweep does with a workspace of half
 * that size.  The call calls no cudaMalloc, cudaFree or allocating library
 * routine.
 *
 * Set-up: the first call on a device (with that device current) looks up
 * the array's device address with cudaGetSymbolAddress and keeps it for that
 * device's context; after a device reset the next call looks it up again.
 * Make the first call on each device before any stream capture begins.  All
 * calls share the one array and it keeps the previous call's contents
 * (everything that must start at zero is cleared by each call), so calls
 * whose work overlaps on the GPU -- on different streams, or from different
 * host threads -- race on it: serialise them.
 */
#define GPTQ_SWEEP_NOALLOC_SCRATCH_BYTES (48u << 20)
gptq_status gptq_q4tp_sweep_noalloc(float* W, int rows, int n, const float* U, const float* hw,
                                    const float* tab, const float* lost, uint8_t* nibbles,
                                    uint8_t* rungs, float* scales, void* stream);

/*
 * The q2tp "placed" rule: 2-bit codes on the levels (q - 1.5) * s, q in 0..3,
 * with the per-(row, group) scale s from a per-row ladder of 31 rungs.
 * [fold page] WGSL q2_level, q2tp_group, host fn sweep_q2tp; [host page]
 * Q2tpRule::Placed, gptq_quantize_q2tp, gptq_quantize_q2tp_dev.
 *
 * gptq_q2tp_place -- the ladder ([host page] gptq_quantize_q2tp_dev: placed
 * from the dead-zeroed weights; the placement function is not on the pages).
 * Reading implemented: each group's scale s*_g is the exact minimiser over
 * s > 0 of sum_t h_t (w_t - (q2_level(w_t/s + 1.5) - 1.5) s)^2 with h = hw
 * clipped at 0 (found among the 33 stationary points of its quadratic
 * pieces, winner recomputed in f64; two scores within 1e-12 * sum h w^2 of
 * each other are a tie, taken by the smaller scale); groups with no channel where h > 0 and
 * w != 0 are left out.  lo = f16(log2 min s*), step = f16(max(0, (log2 max
 * s* - lo)/30)) (0 if min == max), tab[0] = 0, tab[c] = f32(2^(lo + (c-1)
 * step)) for c = 1..31; a row with no group left gets zeros.
 *
 *   W      in  f32 rows*n (dead columns zeroed), n % 32 == 0.
 *   hw     in  f32 n: H_ii (values that are not > 0 count as 0).
 *   tab    out f32 rows*32;  lost out f32 rows*2 = (lo, step).
 *   gscale out f32 rows*n/32 (may be NULL): s*_g, 0 for groups left out.
 */
gptq_status gptq_q2tp_place(const float* W, int rows, int n, const float* hw, float* tab,
                            float* lost, float* gscale, void* stream);

/*
 * gptq_q2tp_group -- the q2tp rung + rounding + in-group feedback rule alone
 * on one 32-column tile of every row ([fold page] WGSL q2tp_group):
 * rung 0 for an all-zero tile, else the lowest of rungs 1..31 with the
 * smallest hw-weighted error of q2_level(w (1/s) + 1.5) (rungs with s <= 0
 * skipped; rung 1 if none scores below 3.4e38); per column q =
 * q2_level(w_j / s + 1.5) (0 if s <= 0), e_j = (w_j - (q - 1.5) s)/U_jj (0 if
 * U_jj <= 0), w_t -= e_j U_jt for t > j.  f32, one rounding per operation.
 *
 *   tile in f32 rows*32; ublk in f32 32*32; hw in f32 32 (clipped at 0);
 *   tab in f32 rows*32.  codes out u8 rows*8 (the tile's 2-bit bytes, see
 *   gptq_q2tp_sweep); rungs out u8 rows; scales out f32 rows; E out f32 rows*32.
 */
gptq_status gptq_q2tp_group(const float* tile, int rows, const float* ublk, const float* hw,
                            const float* tab, uint8_t* codes, uint8_t* rungs, float* scales,
                            float* E, void* stream);

/*
 * gptq_q2tp_sweep -- the column-sequential q2tp GPTQ sweep of W against U
 * ([fold page] sweep_q2tp; [host page] gptq_quantize_q2tp, placed rule,
 * natural column order), with the residuals applied per block of 128
 * columns as in gptq_q4tp_sweep.
 *
 *   W     in/out f32 rows*n (dead columns zeroed); consumed.
 *   U     in  f32 n*n from gptq_fold.  hw in f32 n: H_ii (clipped at 0).
 *   tab   in  f32 rows*32 from gptq_q2tp_place.
 *   codes out u8 rows*n/4: tile (row, group) = 8 bytes at (row*n/32 +
 *         group)*8; column j -> byte j/4, bits 2*(j%4) (the same bytes as
 *         two little-endian u32 words with bits 2*(j%16)).
 *   rungs out u8 rows*n/32; scales out f32 rows*n/32 = tab[row][rung].
 *   ws    >= gptq_sweep_workspace_bytes(rows, n).
 */
gptq_status gptq_q2tp_sweep(float* W, int rows, int n, const float* U, const float* hw,
                            const float* tab, uint8_t* codes, uint8_t* rungs, float* scales,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * gptq_quantize_group_q2tp -- fold + dead-column zeroing + placed ladder +
 * q2tp sweep for one Hessian group ([host page] gptq_fold_dev then
 * gptq_quantize_q2tp_dev).  Arguments as gptq_quantize_group, with the
 * 2-bit plane `codes` (rows*n/4 bytes) in place of the nibbles;
 * ws >= gptq_group_workspace_bytes(rows, n).  Repeated calls are replayed
 * from a captured graph as gptq_quantize_group's are (its own argument sets).
 */
gptq_status gptq_quantize_group_q2tp(const float* H_packed, int n, double lambda, const float* W,
                                     int rows, uint8_t* codes, uint8_t* rungs, float* scales,
                                     float* tab, float* lost, float* U, float* D, float* hdiag,
                                     double* lambda_used, void* ws, size_t ws_bytes, void* stream);

/*
 * gptq_debias -- output debias of a quantized matrix ([host page]
 * q2tp_debias_hessian / q4tp_debias_hessian, GEMM form q2tp_debias_gemm):
 * per row the regression slope b = num/den of the quantized outputs on the
 * original ones, num = (W^ H W^T)_rr, den = (W H W^T)_rr, is removed through
 * the row's f16 lo; codes, rungs and step stay.  The lo update is not on the
 * pages; reading implemented: lo' = f16(lo + log2(den/num)) when num > 0
 * and den > 0 (else lo is kept), the row's rungs rebuilt from (lo', step)
 * (q2tp: rung 0 = 0, rung c = 2^(lo' + (c-1) step); q4tp: 2^(lo' + c step);
 * a row with no non-zero rung keeps its zeros) and every scale set to its
 * rung's new value.  W H on the tensor cores (3xTF32, f32 accumulation
 * drained every 128 of K), the row dots with compensated f32 sums.
 *
 *   bits     2 (q2tp: codes = the 2-bit plane of gptq_q2tp_sweep) or 4
 *            (q4tp: codes = the nibble plane of gptq_q4tp_sweep).
 *   W        in  f32 rows*n: the original weights (dead channels have zero
 *            rows and columns in H, so their weights do not count).
 *   H_packed in  f32 n(n+1)/2: the raw Hessian, as gptq_fold reads it.
 *   codes, rungs in: the sweep's outputs.
 *   tab, lost, scales in/out: the sweep's ladder, (lo, step) and scales;
 *            rewritten for the rows whose slope is positive.
 *   num_den  out f64 rows*2 (may be NULL): num, den per row.
 *   ws       >= gptq_debias_workspace_bytes(rows, n) (dense H as a TF32 pair,
 *            W as a TF32 pair, W H).  Reads back a 4-byte status at the end.
 */
size_t gptq_debias_workspace_bytes(int rows, int n);
gptq_status gptq_debias(int bits, const float* W, int rows, int n, const float* H_packed,
                        const uint8_t* codes, const uint8_t* rungs, float* tab, float* lost,
                        float* scales, double* num_den, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes gptq_quantize_group (and gptq_quantize_group_q2tp) needs. */
size_t gptq_group_workspace_bytes(int rows, int n);

/*
 * gptq_quantize_group -- fold + dead-column zeroing + ladder + sweep for one
 * Hessian group ([host page] run_quantize_gptq_tiled's device path:
 * gptq_fold_dev then gptq_quantize_q4tp_dev).  W is not modified (a zeroed
 * copy lives in the workspace).  U, D, hdiag may be NULL (then they live in
 * the workspace only); otherwise they receive the fold's outputs.  The call
 * returns once its work is done (it reads the pivot flag and the sweep's
 * status back).
 *
 * Repeated calls: the library keeps, per process, the 32 argument sets it
 * saw last (every pointer and size, lambda, the device context and the wait
 * limits).  The second call with a set is captured into a CUDA graph -- one
 * fold attempt at lambda, the ladder, the sweep -- on a stream of the
 * library's own (one per host thread and device), ordered after the caller's work on
 * `stream` by an event, and later calls replay it; the results are the
 * same bit for bit.  If the attempt finds H not positive definite, the call
 * continues on `stream` from the next lambda, as the first call would.
 * Calls made while the caller captures `stream`, or while per-launch
 * profiling records, never capture.  Buffers must stay valid while any call
 * that uses them runs.
 */
gptq_status gptq_quantize_group(const float* H_packed, int n, double lambda, const float* W,
                                int rows, uint8_t* nibbles, uint8_t* rungs, float* scales,
                                float* tab, float* lost, float* U, float* D, float* hdiag,
                                double* lambda_used, void* ws, size_t ws_bytes, void* stream);

/*
 * gptq_build_equilibrated -- the builder step alone ([fold page] build_a):
 * A[i][j] = (H[ii][jj] + delta_ij damp) / (d_ii d_jj), ii = n-1-i, dead
 * channels an identity row/column, damp = lambda * max(mean diag, 1e-12).
 * Writes the lower triangle of the n*n f32 A (upper left untouched) and the
 * signed D.  Uses the fold workspace.
 */
gptq_status gptq_build_equilibrated(const float* H_packed, int n, double lambda, float* A,
                                    float* D, void* ws, size_t ws_bytes, void* stream);

/*
 * Act order ([host page] act_order_perm, permute_sym,
 * gptq_quantize_q4tp_act_order): channels are eliminated in descending H_ii
 * order (Rust total order on f32, ties by index), against the fold operator
 * of H[perm][perm]; every tile's rung is fixed up front ("static groups")
 * and only the codes move.  The static rung is read here as the q4tp rung
 * rule with unit weights on the dead-zeroed original weights (the pages
 * call the converter for it, which they do not show).
 *
 * gptq_act_order_perm   perm (int32 n, out): position a holds channel
 *                       perm[a]; hdiag = raw H_ii (n).
 * gptq_fold_permuted    gptq_fold of H[perm][perm] (entries gathered from
 *                       the packed H): U, D, hdiag in permuted order.
 * gptq_static_rungs     rungs (u8 rows*n/32) and scales (f32) of every
 *                       (row, group) from the dead-zeroed W and its ladder.
 * gptq_q4tp_sweep_act_order  the sweep: W (rows*n, original order, dead
 *                       columns zeroed; not modified), U of the permuted H,
 *                       perm, tab, static rungs -> nibble plane (original
 *                       layout, as gptq_q4tp_sweep writes it).
 * gptq_quantize_group_act_order  all of the above for one group; perm_out
 *                       and U may be NULL.
 */
gptq_status gptq_act_order_perm(const float* hdiag, int n, int* perm, void* stream);
gptq_status gptq_fold_permuted(const float* H_packed, int n, double lambda, const int* perm,
                               float* U, float* D, float* hdiag, double* lambda_used, void* ws,
                               size_t ws_bytes, void* stream);
gptq_status gptq_static_rungs(const float* W, int rows, int n, const float* tab, const float* lost,
                              uint8_t* rungs, float* scales, void* stream);
size_t gptq_sweep_act_order_workspace_bytes(int rows, int n);
gptq_status gptq_q4tp_sweep_act_order(const float* W, int rows, int n, const float* U,
                                      const int* perm, const float* tab, const uint8_t* rungs,
                                      uint8_t* nibbles, void* ws, size_t ws_bytes, void* stream);
size_t gptq_group_act_order_workspace_bytes(int rows, int n);
gptq_status gptq_quantize_group_act_order(const float* H_packed, int n, double lambda,
                                          const float* W, int rows, uint8_t* nibbles,
                                          uint8_t* rungs, float* scales, int* perm_out, float* U,
                                          double* lambda_used, void* ws, size_t ws_bytes,
                                          void* stream);

/*
 * gptq_gram_add -- calibration Hessian accumulation H += X^T X for one window
 * of tokens ([host page] calibration pass: gram_alloc / gram_add_dev, one
 * accumulator per linear input; [fold page] poff: the packed layout).  The
 * pages sum over tokens and keep the token count apart: no normalization.
 *
 *   H_packed in/out f32 n(n+1)/2, upper triangle by rows (as gptq_fold reads).
 *   X        in     f32 T*n row-major (token t, channel i at X[t*n + i]).
 *   T >= 0 tokens (T == 0: nothing to do).  ws >= gptq_gram_workspace_bytes(n)
 *   (a dense n x n scratch plus two n x 4096 operand slices).
 * Products on the tensor cores with the 3xTF32 split, f32 accumulation;
 * reads back a 4-byte status word (stream synchronisation) at the end.
 */
size_t gptq_gram_workspace_bytes(int n);
gptq_status gptq_gram_add(float* H_packed, int n, const float* X, int T, void* ws,
                          size_t ws_bytes, void* stream);

/*
 * Tracing: launch accounting and per-kernel timing.  Every kernel launch of
 * the library is counted; between gptq_profile_start and gptq_profile_stop
 * each launch is also bracketed by a pair of CUDA events recorded on the
 * launching stream (host-side event objects, created once and reused; no
 * device memory).  Single host thread at a time.
 *
 *   gptq_launch_count     kernels launched by the library since it loaded.
 *   gptq_kernel_kinds     number of kernel kinds; gptq_kernel_kind_name(k)
 *                         their names ("fold_gemm", "sweep_gemm", ...).
 *   gptq_profile_select   which kinds record events (bit k = kind k; all
 *                         by default); the others are still counted.  Fewer
 *                         events, less perturbation of the timed launches.
 *   gptq_profile_start    start recording, up to max_launches launches.
 *   gptq_profile_stop     synchronise the recorded events, write per-kind
 *                         total milliseconds and launch counts (host arrays
 *                         of nkinds entries, either may be NULL), stop.
 *                         Returns the kinds written, -2 if max_launches was
 *                         reached (later launches went unrecorded), -1 on a
 *                         CUDA error.
 */
long long gptq_launch_count(void);
int gptq_kernel_kinds(void);
/*
 * gptq_test_set_wait -- test hook for the bounded device waits (the pages
 * have no counterpart: their device path reports a failed pivot through a
 * flag and never waits on another agent).  Every wait inside the
 * tensor-core kernels gives up after wait_ns of device time (0 = the default,
 * 2 s; at most 10 s, else GPTQ_ERR_ARG), stops issuing, drains what it
 * started, frees its tensor memory and sets the status that the calls report
 * as GPTQ_ERR_TIMEOUT.  no_loads = 1 makes the GEMM producers issue no loads
 * at all, so that those waits run out on purpose; no_loads = 0 restores
 * normal work.  Applies to launches made after the call, from any thread;
 * not meant to change while calls are in flight.
 */
gptq_status gptq_test_set_wait(unsigned long long wait_ns, int no_loads);
const char* gptq_kernel_kind_name(int kind);
void gptq_profile_select(unsigned kind_mask);
gptq_status gptq_profile_start(int max_launches);
int gptq_profile_stop(double* ms_by_kind, long long* launches_by_kind, int nkinds);

#ifdef __cplusplus
}
#endif
#endif /* GPTQ_FOLD_H */
