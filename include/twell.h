/*
 * twell.h - C ABI of the GB300 (sm_103a) activation-sparse gated FFN library.
 *
 * The library computes the gated feed-forward block of a ReLU Transformer,
 *     z = x W_g,   h = ReLU(z),   u = x W_u,   y = (h * u) W_d,
 * with the gate activation h held in TwELL (Tile-wise ELLPACK), and the
 * training step over the hybrid (ELL + dense backup) format.
 *
 * Sources ("Sparser, Faster, Lighter Transformer Language Models", summary
 * at gist.science, and the news article "Sakana AI and NVIDIA TwELL boosts
 * LLM training speed by 21.9%"):
 *   - ReLU replaces SiLU so the gate has exact zeros; an L1 term with
 *     coefficient 2e-5 on the FFN activations (news article, recipe list;
 *     paper section 2.A).
 *   - TwELL splits the gate columns into horizontal tiles the width of the
 *     matmul tile and is written in the epilogue of the gate matmul
 *     h_g = ReLU(x W_g), with no separate conversion kernel (paper section
 *     2.B.1; news article, epilogue paragraph).
 *   - One fused kernel does the up and down projections from the TwELL gate,
 *     computing dot products only for nonzeros (paper section 2.B.2).
 *   - Training converts TwELL to a hybrid format (compact ELL rows plus a
 *     dense backup for overflow rows) and runs sparse-to-dense and
 *     dense-to-sparse matmuls forward and backward (paper section 2.B.3).
 *
 * Conventions (every entry point):
 *   - bf16 tensors are passed as uint16_t bit patterns.  Pointers are device
 *     pointers unless stated otherwise.  The caller owns all memory; the
 *     library allocates nothing and never synchronises: all work is enqueued
 *     on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *   - Weights are stored neuron-major, [F][D] row-major: Wg_t = W_g^T,
 *     Wu_t = W_u^T, Wd = W_d.  Activations x, y are [T][D] row-major.
 *   - Arguments are validated on the host before anything is enqueued.  A
 *     failure returns TWELL_ERR_INVALID (or TWELL_ERR_UNSUPPORTED) and
 *     enqueues nothing.  TWELL_ERR_CUDA means a CUDA call failed while
 *     enqueuing; cudaGetLastError() then holds the CUDA error.
 *   - Data-dependent conditions found on the device (a full spill list, a
 *     full dense backup, a wait that timed out) never trap: the kernels OR a
 *     TWELL_FLAG_* bit into *status_dev (a caller-owned device int32 the
 *     library never clears) and the outputs of the affected rows are then
 *     undefined.  Read it after synchronising the stream.
 *   - Alignment: every pointer 16-byte aligned; D % 8 == 0 (rows of 16-byte
 *     multiples); F % 128 == 0; tile == 128.
 */
#ifndef TWELL_H
#define TWELL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TWELL_OK = 0,
  TWELL_ERR_INVALID = 1,      /* bad argument; nothing enqueued */
  TWELL_ERR_UNSUPPORTED = 2,  /* device is not sm_103 or a size limit is exceeded */
  TWELL_ERR_CUDA = 3          /* a CUDA runtime call failed while enqueuing */
} twell_status;

/* Bits OR-ed into *status_dev by the kernels. */
enum {
  TWELL_FLAG_SPILL_FULL = 1,  /* more (row, tile) slices overflowed W than spill_cap */
  TWELL_FLAG_DENSE_FULL = 2,  /* more overflow rows than the hybrid's max_dense */
  TWELL_FLAG_TIMEOUT = 4,     /* a pipeline wait exceeded its bound (about 1 s by default) */
  TWELL_FLAG_RANGE = 8,       /* a value exceeded the fp16 range of an fp16 operand */
  TWELL_FLAG_BOUNDS = 16      /* bounds-checking build only: a gathered or scattered
                                 index fell outside its buffer (access skipped) */
};

#define TWELL_TILE 128

/*
 * TwELL gate activation of a [T][F] matrix (paper section 2.B.1).
 * n_t = F / tile column tiles.  For row t and tile k (columns
 * [k*tile, (k+1)*tile)):
 *   cnt[t*n_t + k]            number of active entries (z > 0), 0..tile
 *   col[(t*n_t + k)*W + s]    local column of slot s (ascending), s < min(cnt, W)
 *   val[(t*n_t + k)*W + s]    z at that column, fp32 (the accumulator's value)
 * Slots at or beyond min(cnt, W) are not written and hold anything.
 * When cnt > W the (row, tile) keeps its first W actives in the slots and its
 * whole fp32 slice ReLU(z) (tile values) in the spill list:
 *   spill_slot[t*n_t + k]     index of that slice, meaningful only where cnt > W;
 *                             an index >= spill_cap means the list was full
 *   spill_rt[s]               t*n_t + k of slice s
 *   spill_val[s*tile + c]     fp32 ReLU(z) of column k*tile + c
 *   *spill_n                  slices requested by the last pack (device int32;
 *                             may exceed spill_cap, then TWELL_FLAG_SPILL_FULL)
 *   block_bits[b*(F/32) + w] optional (may be NULL): bit i of word w is set
 *                             iff column 32*w + i is active (z > 0) in some row
 *                             of the block of rows [128 b, 128 b + 128)
 *                             (every active column counts, spilled or not)
 * Sizes: val [T][n_t][W] float, col [T][n_t][W] uint8, cnt [T][n_t] uint8,
 * spill_slot [T][n_t] int32, spill_rt [spill_cap] int32,
 * spill_val [spill_cap][tile] float, block_bits [ceil(T/128)][F/32] uint32.
 * spill_* may be NULL when spill_cap = 0.  A reader trusts block_bits to
 * describe the same gate as the rest of the TwELL.
 * (The pages leave the value precision open; fp32 keeps the stored gate
 * exact to the accumulator, where bf16 alone would cost up to ~2% of RMS(y).)
 */
typedef struct {
  int32_t T;          /* rows (tokens) */
  int32_t F;          /* columns (d_ff), a multiple of tile */
  int32_t tile;       /* column tile width; must be TWELL_TILE */
  int32_t width;      /* W: slots per (row, tile), 1..tile */
  float* val;
  uint8_t* col;
  uint8_t* cnt;
  int32_t* spill_slot;
  int32_t spill_cap;
  int32_t* spill_n;
  int32_t* spill_rt;
  float* spill_val;
  uint32_t* block_bits;
} twell_t;

/*
 * Gate GEMM with the TwELL epilogue (paper section 2.B.1; news article,
 * epilogue paragraph): z = x W_g with fp32 accumulation on the tensor cores,
 * then, in the same kernel, every (row, tile) slice of z is packed into
 * `*out`.  No dense h is written.
 *   x        [T][D] bf16            Wg_t  [F][D] bf16 (= W_g^T)
 *   out      TwELL with out->T == T, out->F == F; the kernel resets
 *            *out->spill_n to 0 first (stream-ordered) and, when
 *            out->block_bits is not NULL, fills every word of it
 *   z_debug  optional [T][F] fp32 copy of z (NULL to skip), for checking
 *   status_dev  device int32, see TWELL_FLAG_*
 * T may be 0 (nothing enqueued).
 */
twell_status twell_gate_pack(const uint16_t* x, const uint16_t* Wg_t, int32_t T, int32_t D,
                             int32_t F, const twell_t* out, float* z_debug,
                             int32_t* status_dev, void* stream);

/*
 * Decode-sized forward in one call (paper sections 2.B.1 and 2.B.2
 * together): the gate GEMM z = x W_g with its TwELL epilogue, exactly as
 * twell_gate_pack (same `out`, same z_debug), then y = sum over the active
 * entries (t, j) of (h u) W_d[j, :] with u = x_t . W_u[:, j] (fp32).  Up to 8
 * tokens (or d_model > 3072) the projection runs inside the gate kernel: every
 * active entry of z -- slots and spill alike, so nothing is dropped when the
 * spill list is full -- adds its row to y with fp32 atomics.  With more
 * tokens the gate kernel prefetches the active neurons' W_u and W_d rows
 * into L2 and zeroes y while it streams W_g, and the call then runs
 * twell_ffn_fwd's kernel on the TwELL it wrote (whose rules then hold: a
 * missing spill slice is skipped and flagged).  Rows with no active entry
 * get y_t = 0.
 *   x   [T][D] bf16   Wg_t, Wu_t, Wd  [F][D] bf16   y  [T][D] fp32 (written;
 *   zeroed by the call, stream-ordered)   status_dev  device int32 (required)
 * Supports 1 <= T <= 256 with D > 64 (TWELL_ERR_UNSUPPORTED otherwise:
 * use twell_gate_pack + twell_ffn_fwd); D % 8 == 0, all pointers 16-byte
 * aligned.  Repeats agree to fp32 rounding, not bit for bit (atomics).
 */
twell_status twell_ffn_decode(const uint16_t* x, const uint16_t* Wg_t, const uint16_t* Wu_t,
                              const uint16_t* Wd, int32_t T, int32_t D, int32_t F,
                              const twell_t* out, float* y, float* z_debug, int32_t* status_dev,
                              void* stream);

/*
 * Bound, in nanoseconds, on each pipeline wait of the gate kernel launched
 * by later twell_gate_pack calls (process-wide; 0 restores the default of
 * 1e9 ns); returns the previous bound.  A wait that runs out sets
 * TWELL_FLAG_TIMEOUT; the kernel then waits (up to 1 s each) for the TMA
 * loads and MMAs it already issued, frees its tensor memory and returns, so
 * the context stays usable and the TwELL of that call is undefined.  Meant
 * for exercising that path (the paper has no counterpart); a bound of a
 * few nanoseconds makes every call time out.
 */
uint64_t twell_gate_pack_wait_limit(uint64_t ns);

/*
 * Fused up + down projection from a TwELL gate (paper section 2.B.2): for
 * each row t and each stored active entry (j, h), u = x_t . W_u[:, j]
 * (fp32), and y_t += (h u) W_d[j, :] (fp32 accumulation).  Rows with no
 * active entry get y_t = 0.
 *   x   [T][D] bf16, T = h->T      Wu_t, Wd  [F][D] bf16, F = h->F
 *   y   [T][D] fp32 (written; fp32 because a bf16 output alone can exceed a
 *       2e-2 * RMS(y) error where |y| reaches 10 * RMS)
 * A (row, tile) whose spill slice is missing (index >= spill_cap) is skipped
 * and TWELL_FLAG_SPILL_FULL is set.  With few rows (decode batches) a row is
 * split over several warps whose partial sums are added with float atomics
 * into y (zeroed first), so repeated calls agree to fp32 rounding, not bit
 * for bit; with many rows each row is summed by one warp in a fixed order.
 */
twell_status twell_ffn_fwd(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                           const uint16_t* Wd, int32_t D, float* y, int32_t* status_dev,
                           void* stream);

/*
 * Tensor-core variant of twell_ffn_fwd (paper section 2.B.2: up and down
 * projections of the active neurons only, built to keep the tensor cores
 * busy).  Same function, different arithmetic: for each block of 128 rows
 * the union U of the rows' active neurons (h->block_bits when it is not
 * NULL, else built from the slots and spill slices) is gathered, u = x W_u[:, U] is
 * one tcgen05 GEMM (bf16 in, fp32 out), a = h u is rounded to fp16 at each
 * row's own active neurons (0 at the union's other positions), and
 * y = a W_d[U, :] is a second tcgen05 GEMM on fp16 operands (W_d converted
 * from bf16 into the workspace, exactly for |w| >= 2^-14) with fp32
 * accumulation.  The fp16 rounding of h u adds up to 2^-11 |h u| (+ 2^-25)
 * per term to y; fp16 rather than bf16 keeps y within the 2e-2 * RMS bar
 * where a bf16 a (2^-8) did not (30-40 active terms of one row).  A |h u|
 * beyond the fp16 range (65504) sets TWELL_FLAG_RANGE.
 *   x [T][D] bf16, T = h->T, D a multiple of 64;  Wu_t, Wd [F][D] bf16,
 *   F = h->F <= 32768;  y [T][D] fp32 (every row written)
 *   Wd_f16  optional [F][D] fp16 copy of Wd (twell_to_f16); NULL: the call
 *           makes one in the workspace (one extra pass over W_d)
 *   ws: twell_workspace_size(TWELL_WS_FFN_FWD_TC, T, D, F, 0, 0) bytes,
 *       256-byte aligned (per-block unions and position prefixes, the
 *       [T][F] fp16 matrix of a in union order and the fp16 copy of W_d:
 *       about 2 (T + D) F bytes)
 * A (row, tile) whose spill slice is missing is skipped and
 * TWELL_FLAG_SPILL_FULL is set.  Results do not depend on how the work is
 * scheduled: repeated calls agree bit for bit.  T may be 0.
 * Returns TWELL_ERR_UNSUPPORTED for F > 32768, TWELL_ERR_INVALID for a D
 * that is not a multiple of 64 or a workspace that is too small.
 */
twell_status twell_ffn_fwd_tc(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                              const uint16_t* Wd, const uint16_t* Wd_f16, int32_t D, float* y,
                              void* ws, size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * twell_ffn_fwd_tc over blocks of rows grouped by activity: the rows are
 * first ordered by their count of active neurons (a stable sort into eight
 * buckets per octave of the count), then every block of 128 rows in that
 * order is processed as in twell_ffn_fwd_tc (h->block_bits is not read; the
 * blocks' unions are built from the slots and spill slices) and each y row
 * is written to its own token.  A block's union grows with its rows'
 * summed activity in a concave way, so when the per-row activity varies
 * widely (a heavy-tailed batch) the sorted blocks have a much smaller total
 * union and the GEMMs less work; when every row is about equally active
 * the sort and the copy of x in sorted order only add time.  Same
 * arguments, results and errors as twell_ffn_fwd_tc; the workspace is
 * twell_workspace_size(TWELL_WS_FFN_FWD_TC_SORTED, T, D, F, 0, 0) bytes (that
 * of twell_ffn_fwd_tc plus the row order and a copy of x: + 2 T D + 5 T
 * bytes and a little more).  Rows are summed in an order fixed by the data,
 * so repeated calls agree bit for bit.
 */
twell_status twell_ffn_fwd_tc_sorted(const uint16_t* x, const twell_t* h, const uint16_t* Wu_t,
                                     const uint16_t* Wd, const uint16_t* Wd_f16, int32_t D,
                                     float* y, void* ws, size_t ws_bytes, int32_t* status_dev,
                                     void* stream);

/*
 * fp16 copy of bf16 values (for the W_d operand of twell_ffn_fwd_tc, made
 * once for weights that do not change between calls): dst[i] = fp16(src[i]),
 * round to nearest; exact for |v| >= 2^-14 (bf16 has fewer significant
 * bits); |v| > 65504 becomes inf and sets TWELL_FLAG_RANGE.
 *   src, dst  device arrays of n elements, 16-byte aligned, n a multiple of 8
 */
twell_status twell_to_f16(const uint16_t* src, uint16_t* dst, size_t n, int32_t* status_dev,
                          void* stream);

/*
 * Hybrid training format (paper section 2.B.3): rows whose every tile count
 * is at most the ELL capacity C stay in a compact ELL matrix; the other
 * ("overflow") rows go to a dense backup.  Both lists are in ascending token
 * order.  Reading: a row overflows iff some tile count exceeds C (a count of
 * exactly C stays in ELL).
 *   *n_ell, *n_dense          device int32 row counts (n_dense is the true
 *                             number of overflow rows; rows past max_dense get
 *                             no dense row and TWELL_FLAG_DENSE_FULL is set)
 *   row_map[t]                i >= 0: ELL row i;  i < 0: dense row -(i+1)
 *   ell_rows[i]               token of ELL row i, i < n_ell
 *   ell_cnt[i*n_t + k]        count of ELL row i in tile k (<= C)
 *   ell_col/ell_val[(i*n_t + k)*C + s]   its entries, ascending, s < count;
 *                             padding slots (s >= count) hold column 0xFF
 *   dense_rows[i]             token of dense row i, i < min(n_dense, max_dense)
 *   dense_h[i*F + j]          fp32 ReLU(z) of that token (zeros where inactive)
 * Sizes: row_map, ell_rows [T] int32; ell_cnt [T][n_t] uint8;
 * ell_col [T][n_t][C] uint8; ell_val [T][n_t][C] float (T rows reserved since
 * every row may be an ELL row); dense_rows [max_dense] int32;
 * dense_h [max_dense][F] float.
 */
typedef struct {
  int32_t T;
  int32_t F;
  int32_t tile;       /* must be TWELL_TILE */
  int32_t cap;        /* C: ELL slots per (row, tile), 1..tile */
  int32_t max_dense;  /* rows reserved for the dense backup, >= 0 */
  int32_t* n_ell;
  int32_t* n_dense;
  int32_t* row_map;
  int32_t* ell_rows;
  float* ell_val;
  uint8_t* ell_col;
  uint8_t* ell_cnt;
  int32_t* dense_rows;
  float* dense_h;
} hybrid_t;

/*
 * TwELL -> hybrid conversion (paper section 2.B.3: a custom kernel converts
 * TwELL to the hybrid format).  Reads the TwELL `h` (slots and spill) and
 * fills `out` (out->T == h->T, out->F == h->F; C = out->cap may differ from
 * h->width: entries beyond W come from the spill slices).  Row lists and
 * counts are produced on the device; nothing is read back.  A (row, tile)
 * that needs its spill slice when the TwELL's spill list had no room for it
 * is stored empty (ELL count 0, every slot padding; zeros in a dense row)
 * and TWELL_FLAG_SPILL_FULL is set.
 */
twell_status twell_to_hybrid(const twell_t* h, const hybrid_t* out, int32_t* status_dev,
                             void* stream);

/* Workspace operations for twell_workspace_size. */
enum {
  TWELL_WS_HYBRID_FWD = 1,
  TWELL_WS_HYBRID_BWD = 2,
  TWELL_WS_HYBRID_FWD_TC = 3,
  TWELL_WS_HYBRID_BWD_TC = 4,
  TWELL_WS_FFN_FWD_TC = 5,        /* twell_ffn_fwd_tc; cap and max_dense are ignored */
  TWELL_WS_FFN_FWD_TC_SORTED = 6  /* twell_ffn_fwd_tc_sorted; cap and max_dense ignored */
};

/*
 * Bytes of device workspace `op` needs for a hybrid of T rows, width d_model
 * D, F columns, ELL capacity C and max_dense dense rows (0 on bad
 * arguments).  The workspace is scratch the call overwrites; it must be
 * 256-byte aligned and not shared by calls that may overlap on the GPU.
 */
size_t twell_workspace_size(int32_t op, int32_t T, int32_t D, int32_t F, int32_t cap,
                            int32_t max_dense);

/*
 * Hybrid training forward (paper section 2.B.3: dense-to-sparse and
 * sparse-to-dense matmuls over the hybrid format).
 *   ELL rows (CUDA cores): u = x_t . W_u[:, j] at every ELL entry, saved in
 *     u_ell (same layout as ell_val), and y_t = sum_j (h u) W_d[j, :].
 *   Dense rows (tensor cores): U = X_ov W_u, saved in U_dense [max_dense][F]
 *     fp32; y_ov = (H_ov * U) W_d with the fp32 product split into bf16 hi
 *     and lo halves (two MMAs), so the bf16 operand adds no rounding beyond
 *     about 2^-17 relative.
 *   x [T][D] bf16; Wu_t, Wd [F][D] bf16; y [T][D] fp32 (every row written,
 *   dense rows past max_dense excepted); u_ell [T][n_t][C] fp32;
 *   ws: twell_workspace_size(TWELL_WS_HYBRID_FWD, ...) bytes (may be NULL
 *   when max_dense == 0).  Dense rows of y sum split-K partial products with
 *   atomics, so they agree across calls to fp32 rounding, not bit for bit.
 */
twell_status hybrid_ffn_fwd(const uint16_t* x, const hybrid_t* h, const uint16_t* Wu_t,
                            const uint16_t* Wd, int32_t D, float* y, float* u_ell,
                            float* U_dense, void* ws, size_t ws_bytes, int32_t* status_dev,
                            void* stream);

/*
 * Hybrid training backward with the L1 term (paper section 2.B.3; L1
 * coefficient from the news article's recipe list).  For the loss
 * L(y) + l1_coeff * sum(h), with dy = dL/dy [T][D] fp32 and a = h * u:
 *   da = dy W_d^T;  du = da h;  dz = da u + l1_coeff at active entries;
 *   dx = dz W_g^T + du W_u^T;  dW_g^T = dz^T x;  dW_u^T = du^T x;
 *   dW_d = a^T dy.
 * ELL rows run on the CUDA cores (dense-to-sparse da, sparse-to-dense dx,
 * per-neuron records for the weight gradients); dense rows run on the tensor
 * cores with fp32 operands split into bf16 hi and lo halves.
 *   u_ell, U_dense   as written by hybrid_ffn_fwd for the same hybrid
 *   dx [T][D] fp32 (written);  dWg_t, dWu_t, dWd [F][D] fp32 (overwritten,
 *   not accumulated, in the weights' neuron-major layout)
 *   ws: twell_workspace_size(TWELL_WS_HYBRID_BWD, ...) bytes
 * The weight gradients sum per-neuron records in an order set by atomics,
 * and dense rows sum split-K partial products with atomics, so repeated
 * calls agree to fp32 rounding, not bit for bit.
 */
twell_status hybrid_ffn_bwd(const uint16_t* x, const hybrid_t* h, const float* u_ell,
                            const float* U_dense, const uint16_t* Wg_t, const uint16_t* Wu_t,
                            const uint16_t* Wd, int32_t D, const float* dy, float l1_coeff,
                            float* dx, float* dWg_t, float* dWu_t, float* dWd, void* ws,
                            size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * Tensor-core variants of hybrid_ffn_fwd / hybrid_ffn_bwd (the paper's
 * hybrid matmuls of section 2.B.3 mapped onto tcgen05 for activation
 * densities at which every 128-token block touches every 128-neuron tile, so
 * CUDA-core gathers of neuron rows cost more than dense tiles).  Same
 * arguments, outputs and dense-row handling as the CUDA-core entry points;
 * the ELL rows change:
 *   dense-to-sparse products (u, and da in the backward) are full tensor-core
 *   tiles X_ell W_u and dY_ell W_d^T of which only the ELL entries are kept;
 *   sparse-to-dense products (y, dx, dW_g^T, dW_u^T, dW_d) expand the ELL
 *   values tile by tile in shared memory into fp16 operands.
 * Apart from x and W_u in u (bf16, exact), every tensor-core operand of the
 * ELL rows is fp16 (relative rounding up to 2^-11): h u, W_d in y; and in
 * the backward x, the weights and, multiplied by a power of two s that puts
 * max(max |dy|, 2^-14 l1_coeff) in [0.5, 1), dy, dz and du (the fp32
 * products are divided by s again, which rounds nothing); dy in da and dz in
 * dx also carry an fp16 low half (a bias-like column of W_g sums a token's
 * dz, and every da of a token shares the token's dy rounding, into one
 * element of dx).  Weights and the
 * gathered rows are converted into the workspace by each call.  A value
 * beyond the fp16 range sets TWELL_FLAG_RANGE (the results are then not
 * meaningful).  Accumulation is fp32; results differ from the CUDA-core
 * entry points by that rounding.  Requires
 * D % 64 == 0 and C in {16, 32}; other shapes return TWELL_ERR_UNSUPPORTED.
 * Deterministic for the ELL rows (no atomics); dense rows as above.
 *   ws: twell_workspace_size(TWELL_WS_HYBRID_FWD_TC / _BWD_TC, ...) bytes.
 */
twell_status hybrid_ffn_fwd_tc(const uint16_t* x, const hybrid_t* h, const uint16_t* Wu_t,
                               const uint16_t* Wd, int32_t D, float* y, float* u_ell,
                               float* U_dense, void* ws, size_t ws_bytes, int32_t* status_dev,
                               void* stream);
twell_status hybrid_ffn_bwd_tc(const uint16_t* x, const hybrid_t* h, const float* u_ell,
                               const float* U_dense, const uint16_t* Wg_t, const uint16_t* Wu_t,
                               const uint16_t* Wd, int32_t D, const float* dy, float l1_coeff,
                               float* dx, float* dWg_t, float* dWu_t, float* dWd, void* ws,
                               size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * hybrid_ffn_fwd with no workspace argument, for callers that cannot
 * allocate device memory themselves (a loop whose memory budget is fixed up
 * front, a host program without access to a device allocator, code that must
 * not call cudaMalloc because it can synchronise the device).  The paper has
 * no counterpart: this is a packaging of hybrid_ffn_fwd, with the same
 * arguments, results and errors apart from the workspace.
 *   The workspace is a 64 MiB device array inside this library, held on
 *   every GPU that loads it until the process exits.  A hybrid whose
 *   forward workspace (twell_workspace_size(TWELL_WS_HYBRID_FWD, ...)) is
 *   larger returns TWELL_ERR_UNSUPPORTED and enqueues nothing.
 *   The first call on a device looks up the array's device address (with
 *   that device current) and caches it with the device's current context;
 *   make that first call before any stream capture.  After the context is
 *   destroyed and created again (cudaDeviceReset), the array lives at a new
 *   address: the next call sees the new context and looks it up again, so
 *   it too belongs outside stream capture.  The entry point allocates
 *   nothing.
 *   All calls share the array: calls that may overlap on the GPU race.
 */
twell_status hybrid_ffn_fwd_noalloc(const uint16_t* x, const hybrid_t* h, const uint16_t* Wu_t,
                                    const uint16_t* Wd, int32_t D, float* y, float* u_ell,
                                    float* U_dense, int32_t* status_dev, void* stream);

/*
 * FP32 FMA throughput probe (a measurement helper; the paper has no
 * counterpart).  Launches, on `stream`, one grid of two 512-thread CTAs per
 * SM in which every thread runs 16 independent register-resident chains
 * acc = acc * a + b for `iters` rounds: scalar fp32 FMAs (packed = 0) or
 * packed two-lane fma.rn.f32x2 (packed != 0, the form the CUDA-core kernels
 * use).  The caller times the launch with CUDA events; the work is
 * 2 * 16 * iters * (*threads) flops.  `out` (device, 16-byte aligned,
 * out_len >= *threads floats) receives one sum per thread; `*threads` (host)
 * is set before the launch.  TWELL_ERR_INVALID if out_len is too small.
 */
twell_status twell_probe_fma(int32_t packed, int32_t iters, float* out, size_t out_len,
                             int64_t* threads, void* stream);

/* Human-readable name of a status code (static storage). */
const char* twell_status_string(twell_status s);

/* Library version, (major << 16) | minor. */
int32_t twell_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TWELL_H */
