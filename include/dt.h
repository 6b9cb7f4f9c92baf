/*
 * dt.h - C ABI of the chunk-centric fused AllGather-GEMM, GEMM-ReduceScatter,
 *        GEMM-AllReduce and GEMM-AllToAll for one GB300 (sm_103a).
 *
 * What is computed (DITRON page, section 4 "支持的并行策略": tensor parallelism overlaps
 * AllGather with GEMM and GEMM with ReduceScatter; Triton-distributed talk, "GEMM
 * ReduceScatter" paragraph):
 *   AllGather-GEMM     C   = concat_rows(A_0 .. A_{W-1}) * B
 *   GEMM-ReduceScatter out_s = rows [s*M/W, (s+1)*M/W) of  sum_q A_q * B_q
 *   GEMM-AllReduce     out_r = sum_q A_q * B_q  (every rank)
 *   GEMM-AllToAll      out_h = rows stacked by source q of columns [h*N/W, (h+1)*N/W) of
 *                              A_q * B_q  (sequence parallelism, section 4 "序列并行SP")
 * W tensor-parallel ranks are emulated as W "virtual ranks" whose buffers live in the
 * one GPU's HBM.  The user-facing signature is the local GEMM's plus rank and world size
 * (AutoOverlap page, section 3: the fused operator keeps the local kernel's signature and
 * adds rank / world size / mesh).
 *
 * How (AutoOverlap page, sections 4-5; DITRON page, section 3.2):
 *   - communication moves in chunks of `chunk_rows` rows; a per-chunk ready flag flips
 *     when a chunk has landed (chunk abstraction, P2P pull for AllGather, push for
 *     ReduceScatter);
 *   - one persistent tcgen05 GEMM consumes tiles in the rank-aware swizzle order
 *     (gather mode: own rank first, remote chunks in arrival order, tiles that straddle
 *     ranks after the chunks they need; scatter mode: the next rank's rows first, the
 *     own block last) and waits per tile only for the chunks that tile reads;
 *   - the chunk transfer runs on the copy engine, on in-kernel TMA bulk copies, or on
 *     vectorised loads/stores (AutoOverlap page, Table 2 / Fig. 7);
 *   - GEMM-ReduceScatter: a reduction unit is the part of a chunk that one m-tile covers,
 *     times one column tile; its W partial tiles are folded into an fp32 running sum in the
 *     fixed source order q = 0, 1, ..., W-1 (the order the schedule produces them: the
 *     virtual ranks run one after another, each in its own scatter order; a partial that
 *     arrives early waits in a park slot) and rounded once, so results do not depend on
 *     tile order, chunk size or backend.
 *
 * Conventions
 *   - Matrices are row-major with explicit leading dimensions in ELEMENTS.
 *   - Inputs are bf16.  Outputs are bf16 (round to nearest even) or fp32.
 *   - All pointers named "device" are CUDA device pointers on the current device, 16-byte
 *     aligned; leading dimensions are multiples of 8 elements (16-byte TMA strides).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous
 *     and stream-ordered; inputs must stay unchanged, and outputs and the workspace
 *     untouched, until the stream has passed the call.
 *   - The caller owns every buffer, including the workspace.  The library never allocates
 *     device memory.  It keeps a small host-side record per workspace pointer (call epoch,
 *     which plan is resident) and, once per device, a side stream and two events for the
 *     copy-engine backend.
 *   - Errors in the arguments are returned synchronously and nothing is launched.  Errors
 *     found on the device (a bounded wait that ran out) are written to the workspace's
 *     error word and returned by dt_check(); every device wait is bounded by
 *     `timeout_us`, after which the kernel records the error and exits cleanly.
 *   - No C++ exception crosses this boundary.
 */
#ifndef DT_H_
#define DT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DT_MAX_WORLD 16

typedef enum {
  DT_OK = 0,
  DT_ERR_INVALID = 1,      /* bad argument (message: dt_last_error())                    */
  DT_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement               */
  DT_ERR_TIMEOUT = 3,      /* a bounded device wait ran out (from dt_check)               */
  DT_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed                         */
  DT_ERR_WORKSPACE = 5     /* workspace missing, misaligned or smaller than required      */
} dt_status;

typedef enum {
  DT_XFER_AUTO = 0,        /* pick per chunk size                                          */
  DT_XFER_COPY_ENGINE = 1, /* host-issued cudaMemcpy2DAsync + stream flag write per chunk  */
  DT_XFER_TMA = 2,         /* in-kernel cp.async.bulk, global -> shared -> global          */
  DT_XFER_LDST = 3,        /* in-kernel 16-byte vector loads/stores                        */
  DT_XFER_TMA_TILE = 4     /* AllGather-GEMM only: every compute CTA pulls exactly the A rows
                              of its own tiles from the owning shard into its shared-memory
                              operand ring with TMA, and its MMAs wait on that ring's
                              mbarriers (no gather buffer, no global flags); needs every
                              128-row m-tile inside one shard: (M/W) % 128 == 0             */
} dt_xfer;

typedef enum { DT_BF16 = 0, DT_F32 = 1 } dt_dtype;

typedef enum { DT_OP_AG_GEMM = 0, DT_OP_GEMM_RS = 1, DT_OP_GEMM_AR = 2, DT_OP_GEMM_A2A = 3 } dt_op;

/* Problem description shared by every call.  Fill with dt_args_default() first. */
typedef struct dt_args {
  int32_t world_size;  /* W, 1..DT_MAX_WORLD                                               */
  int32_t rank;        /* AllGather-GEMM: the rank whose view is computed (0..W-1);
                          its own shard is "local", the other W-1 are "remote".  RS: unused */
  int64_t m;           /* rows: gathered M for AG, M for RS, W x rows per rank for A2A;
                          M % W == 0                                                       */
  int64_t n;           /* columns of B and C; multiple of 8 (A2A: N/W multiple of 8)       */
  int64_t k;           /* AG: full K (multiple of 8); RS: K per rank; A2A: K               */
  int64_t chunk_rows;  /* rows per communication chunk, >= 1                               */
  int32_t swizzle;     /* 1: rank-aware swizzle order; 0: naive order (all ranks tile 0)   */
  int32_t backend;     /* dt_xfer, AllGather chunk transfer                                */
  int32_t out_dtype;   /* dt_dtype of C / out_s                                            */
  int32_t tile_m;      /* rows of a tile: 128 (one CTA, tcgen05 cta_group::1), 256 (a cluster
                          of two CTAs on two SMs, cta_group::2: each stages 128 rows of A and
                          half of the 256 columns of B, 6 pipeline stages),
                          0 = 256 when that leaves at least 76 tiles (one per SM pair) and
                          copy_ctas is even, else 128; copy_ctas must be a multiple of
                          tile_m / 128                                                      */
  int32_t tile_n;      /* 0 or 256                                                         */
  int32_t group;       /* m-tiles per band of the in-chunk raster; 0 = 8                   */
  int64_t lda;         /* AG: of every shard; RS: of every A_q   (0 = K)                   */
  int64_t ldb;         /* of B / every B_q                       (0 = N)                   */
  int64_t ldc;         /* of C / every out_s (0 = N); A2A: of every out_h (0 = N/W)        */
  int64_t timeout_us;  /* bound of every device wait; 0 = 2 s (env DT_WAIT_TIMEOUT_US)     */
  int32_t num_sms;     /* persistent grid size; 0 = all SMs                                */
  int32_t copy_ctas;   /* AG with DT_XFER_TMA / DT_XFER_LDST: CTAs of the grid that only move
                          chunks (dedicated SMs); 0 = transfer warps inside every compute CTA
                          (co-located).  AutoOverlap page section 5.3, lowerings 2-5.        */
  int32_t act;         /* AG only: dt_act applied to the fp32 result before it is stored     */
  int32_t col_band;    /* AllGather, ReduceScatter / AllReduce tile order: column tiles per
                          column band (the bands run one after another, each repeating the
                          gather order over every chunk, or rank q's scatter order over every
                          destination); 0 = automatic: one band when B (K x N bf16) fits in
                          32 MiB, else the fewest equal bands whose share of B does; >= Tn:
                          one band.  AllToAll: unused                                       */
} dt_args;

typedef enum { DT_ACT_NONE = 0, DT_ACT_GELU_TANH = 1, DT_ACT_SILU = 2 } dt_act;

/* Fill `a` with defaults: W=1, rank 0, swizzle on, AUTO backend, bf16 output, automatic tile
 * rows (tile_m = 0) x 256 columns, group 8.  Sizes are zero and must be set by the caller. */
void dt_args_default(dt_args* a);

/* Library version (major*10000 + minor*100 + patch). */
int dt_version(void);

/* sizeof(dt_args) as compiled into the library, for binding layout checks. */
size_t dt_sizeof_args(void);

/* Human-readable name of a status. Never NULL. */
const char* dt_status_string(dt_status s);

/* Message describing the last DT_ERR_INVALID / DT_ERR_UNSUPPORTED / DT_ERR_CUDA of the
 * calling thread ("" if none).  Valid until the thread's next call. */
const char* dt_last_error(void);

/* Bytes of device workspace that `op` (dt_op) needs for `a`; 0 if `a` is invalid.
 * AG: control block + per-chunk flags/counters + tile order + the gather buffer
 *     (M x K bf16).  RS / AR: control block + per-unit words + tile order + the fp32
 *     running sums (M x N) and park slots (W-1 per destination, M/W x N each).
 *     A2A: control block + per-chunk counters and flags + tile order. */
size_t dt_workspace_size(const dt_args* a, int op);

/* Zero the control block of a workspace laid out for (a, op) on `stream` and forget the
 * library's record of it.  Optional: the first call that sees a workspace (or a changed
 * layout) does the same. */
dt_status dt_workspace_init(const dt_args* a, int op, void* workspace, size_t ws_bytes,
                            void* stream);

/* Fused AllGather-GEMM, rank a->rank's view.
 *   a_shards : host array of W device pointers; shard s is A_s [M/W x K] bf16, ld = lda
 *   b        : device pointer, B [K x N] bf16, ld = ldb
 *   c        : device pointer, C [M x N] (out_dtype), ld = ldc
 *   workspace: device pointer of >= dt_workspace_size(a, DT_OP_AG_GEMM) bytes, 256-byte
 *              aligned, used by one call at a time.
 * Rows of shard s are gathered into the workspace chunk by chunk (own rank first, then
 * r+1, r+2, ...), each chunk's ready flag is released, and the persistent GEMM waits per
 * tile for the chunks of its rows (DITRON page section 3.2 "Gather模式").  With
 * DT_XFER_TMA_TILE there is no gather buffer and no flag: each tile's A rows come straight
 * from the shard that owns them into the consuming CTA's shared memory, synchronised by the
 * pipeline's mbarriers (AutoOverlap page, section 5.3: the co-located lowering coordinates
 * communication and computation on one SM through shared-memory barriers); the tile order
 * still visits the own rank's rows first and then rank r+1, r+2, ...  With W == 1 there
 * is nothing to gather and the GEMM reads the one shard in place (a plain GEMM).  K == 0
 * writes zeros; M == 0 or N == 0 does nothing. */
dt_status dt_ag_gemm(const void* const* a_shards, const void* b, void* c,
                     void* workspace, size_t ws_bytes, const dt_args* a, void* stream);

/* Fused GEMM-ReduceScatter over all W virtual ranks.
 *   a   : host array of W device pointers, A_q [M x K] bf16 (K = per-rank K), ld = lda
 *   b   : host array of W device pointers, B_q [K x N] bf16, ld = ldb
 *   out : host array of W device pointers, out_s [M/W x N] (out_dtype), ld = ldc
 * Every tile (q, i, n) is one partial product.  For each unit (rows of m-tile i inside one
 * chunk, column tile n) the partials are folded in the fixed source order q = 0..W-1 (the
 * virtual ranks run one after another, each sending to rank q+1 first and keeping its own
 * block for last, so each unit receives them in that order): a tile whose partial is next
 * in order adds it to the fp32
 * running sum (the last one rounds into out_s); one that arrives early parks it, and whoever
 * advances the unit past it folds it (notify through one atomic word per unit; nobody
 * waits).  DITRON page section 3.2 "Scatter模式"; Triton-distributed talk, notify/wait of
 * the GEMM-ReduceScatter example. */
dt_status dt_gemm_rs(const void* const* a, const void* const* b, void* const* out,
                     void* workspace, size_t ws_bytes, const dt_args* a_args, void* stream);

/* Fused GEMM-AllReduce over all W virtual ranks (DITRON page, sections 4 and 5.1: GEMM-AR,
 * the third tensor-parallel overlap kernel).  Same inputs, schedule and fixed-order running
 * sums as dt_gemm_rs; the last fold of each unit writes its rows, rounded once, at their
 * global row into every rank's output, so every rank receives all of S = sum_q A_q * B_q.
 *   out : host array of W device pointers, out_r [M x N] (out_dtype), ld = ldc.  If all W
 *         pointers are equal the result is written once.
 * Workspace: dt_workspace_size(a, DT_OP_GEMM_AR) (the same layout as the ReduceScatter). */
dt_status dt_gemm_ar(const void* const* a, const void* const* b, void* const* out,
                     void* workspace, size_t ws_bytes, const dt_args* a_args, void* stream);

/* Fused GEMM-AllToAll over all W virtual ranks (sequence parallelism: DITRON page, section 4
 * "序列并行SP: GEMMAllToAll", section 4.2 weak scaling with a fixed sequence length per rank).
 * Rank q holds its M/W sequence rows A_q and computes Y_q = A_q * B_q (N = W*Nw columns, e.g.
 * the attention heads of all ranks, block h being those that rank h owns); the all-to-all
 * gives rank h columns [h*Nw, (h+1)*Nw) of every Y_q, stacked by source rank:
 *     out_h[q*M/W + r, c] = Y_q[r, h*Nw + c].
 *   a   : host array of W device pointers, A_q [M/W x K] bf16, ld = lda
 *   b   : host array of W device pointers, B_q [K x N] bf16, ld = ldb (a replicated weight
 *         passes the same pointer W times)
 *   out : host array of W device pointers, out_h [M x N/W] (out_dtype), ld = ldc (0 = N/W)
 * Requires N % W == 0 and (N/W) % 8 == 0.  Column tiles never cross a destination's block;
 * every tile's epilogue stores its rows straight into out_h (push, scatter mode: rank q
 * computes destination q+1's block first and its own last, chunk by chunk in row order; the
 * W virtual source ranks run one after another) and
 * counts itself on chunk (h, q, j) = rows [j*chunk_rows, ..) of source q; the count's last
 * tile releases that chunk's ready flag (notify).  Results do not depend on the order, chunk
 * size or group width (each output is one product).  Workspace:
 * dt_workspace_size(a, DT_OP_GEMM_A2A) (control block, counters, flags, tile order only).
 * K == 0 writes zeros; M == 0 or N == 0 does nothing. */
dt_status dt_gemm_a2a(const void* const* a, const void* const* b, void* const* out,
                      void* workspace, size_t ws_bytes, const dt_args* a_args, void* stream);

/* The AllToAll's chunk signals after the last dt_gemm_a2a call on `workspace`: synchronises
 * `stream`, then copies the W*W*nC ready flags and completion counters, index
 * (h*W + q)*nC + j with nC = ceil((M/W)/chunk_rows), to the host arrays `flags` and
 * `counts` (either may be NULL), and the call's epoch to *epoch (may be NULL).  After a
 * completed call every flag equals the epoch and every counter is back to 0.  `len` must
 * equal W*W*nC. */
dt_status dt_a2a_signals(const dt_args* a, void* workspace, void* stream, uint32_t* flags,
                         uint32_t* counts, int64_t len, uint32_t* epoch);

/* Tensor-parallel feed-forward block, AllGather + ReduceScatter form, over W virtual ranks
 * (DITRON page, section 5.1 "FFN模块"; Triton-distributed talk: the AllGather-GEMM feeds the
 * GEMM-ReduceScatter).  Rank q holds column block q of W1 (F_r = F/W columns) and W2_q.
 *   1. h = act(AllGather(x) * W1), all ranks' blocks at once (every rank gathers the same X):
 *      dt_ag_gemm with `ag` (m = M, k = model dim, n = W*F_r, act, out_dtype bf16, ldc = n).
 *   2. out_s = rows s of sum_q h[:, q*F_r .. (q+1)*F_r) * W2_q: dt_gemm_rs with `rs`
 *      (m = M, k = F_r, n = N, lda = W*F_r), A_q = h + q*F_r.
 *   x_shards : W device pointers [M/W x K] bf16;  w1 : [K x W*F_r] bf16;
 *   w2       : W device pointers [F_r x N] bf16;  h : [M x W*F_r] bf16 (written, then read);
 *   out      : W device pointers [M/W x N].
 * Requires ag.world_size == rs.world_size, ag.m == rs.m, ag.n == W * rs.k, rs.k % 8 == 0. */
dt_status dt_ffn_ag_rs(const void* const* x_shards, const void* w1, const void* const* w2,
                       void* h, void* const* out, void* ws_ag, size_t ws_ag_bytes, void* ws_rs,
                       size_t ws_rs_bytes, const dt_args* ag, const dt_args* rs, void* stream);

/* AllGather alone: the chunk transfer of dt_ag_gemm without the GEMM (Triton-distributed
 * talk, "AllGather" producer side; AutoOverlap page, section 4: a P2P op defined at the
 * destination pulls a chunk; DITRON page, section 3.1: device-level chunks move by DMA-style
 * getmem).  out = concat_rows(A_0, .., A_{W-1}), [M x K] bf16 with leading dimension
 * a->ldc (0 = K); every shard, the own one included, is copied chunk by chunk (chunk_rows
 * rows, ragged last chunk) in the AllGather's transfer order (own rank first when swizzle is
 * on, then rank+1, ..).  Backends:
 *   DT_XFER_COPY_ENGINE : one (2-D) copy per chunk on `stream`; any ldc.
 *   DT_XFER_TMA / LDST  : one launch of the fused kernel with no GEMM tiles, every CTA (all
 *                         SMs, or a->num_sms) running the transfer workers (6 TMA bulk-copy
 *                         threads moving 32 KiB pieces, or 8 vector ld/st warps, per CTA; the
 *                         environment variables DT_COPY_PIECE (8192, 16384, 32768) and
 *                         DT_COPY_BUFS (buffers per TMA worker, 1-4) override the TMA
 *                         workers' piece size and depth); each chunk's ready flag in
 *                         the workspace is released with the call's epoch.  Needs ldc == K
 *                         (rows land back to back).
 *   DT_XFER_AUTO        : the AllGather-GEMM's rule (copy engine for chunks of >= 8 MiB, else
 *                         TMA), and the copy engine whenever ldc != K.
 * Uses world_size, rank, M, K, chunk_rows, swizzle, backend, lda, ldc, num_sms; N, ldb,
 * out_dtype, tile_m, act and copy_ctas are ignored.  Workspace: dt_workspace_size(a,
 * DT_OP_AG_GEMM) with any N >= 8 suffices (its gather area is not used).  Inputs and `out`
 * must not overlap.  M == 0 or K == 0 does nothing. */
dt_status dt_allgather(const void* const* a_shards, void* out, void* workspace, size_t ws_bytes,
                       const dt_args* a, void* stream);

/* Kernel-level-overlap baselines with the same arguments and results (AutoOverlap page,
 * section 2.1 / Fig. 2(b)): AG = per-chunk copies on a second stream and one launch of the
 * same GEMM per chunk, gated by events; RS = one GEMM launch per destination block writing
 * fp32 partials, then a separate reduction kernel on a second stream. */
dt_status dt_ag_gemm_kernel_overlap(const void* const* a_shards, const void* b, void* c,
                                    void* workspace, size_t ws_bytes, const dt_args* a,
                                    void* stream);
dt_status dt_gemm_rs_kernel_overlap(const void* const* a, const void* const* b,
                                    void* const* out, void* workspace, size_t ws_bytes,
                                    const dt_args* a_args, void* stream);
dt_status dt_gemm_ar_kernel_overlap(const void* const* a, const void* const* b,
                                    void* const* out, void* workspace, size_t ws_bytes,
                                    const dt_args* a_args, void* stream);
/* GEMM-AllToAll baseline: W GEMM launches, step d computing on every rank q the column
 * block of destination (q + d + 1) mod W into the rank's own buffer y_q, each followed on a
 * second stream by the W copy-engine copies of that step's blocks into out_h; the copies of
 * step d overlap the GEMM of step d+1.
 *   y : host array of W device pointers, y_q [M/W x N] (out_dtype), ld = N, scratch owned
 *       by the caller (each rank's local GEMM output). */
dt_status dt_gemm_a2a_kernel_overlap(const void* const* a, const void* const* b,
                                     void* const* y, void* const* out, void* workspace,
                                     size_t ws_bytes, const dt_args* a_args, void* stream);

/* Tiles of the execution order of `op` for `a` (-1 if `a` is invalid), the rows of one
 * tile (128 or 256, tile_m resolved), and the column tiles per column band of the
 * AllGather / ReduceScatter / AllReduce order (col_band resolved; Tn for the AllToAll). */
int64_t dt_tile_count(const dt_args* a, int op);
int32_t dt_tile_rows(const dt_args* a, int op);
int32_t dt_col_band(const dt_args* a, int op);

/* Tile execution order of `op` for `a` computed on the host: order[p] is the tile run at
 * position p.  AG tile id = i*Tn + n; RS / AR tile id = (q*Tm + i)*Tn + n, with
 * Tm = ceil(M/tile_m), Tn = ceil(N/tile_n); A2A tile id = (q*Tm + i)*Tn + h*Tnw + c with
 * Tm = ceil((M/W)/tile_m), Tnw = ceil((N/W)/tile_n), Tn = W*Tnw; tile_m as resolved by
 * dt_tile_rows.  `len` must equal dt_tile_count.
 * (DITRON page section 3.2: swizzle_func maps the original tile id to the new one.) */
dt_status dt_swizzle_plan(const dt_args* a, int op, int32_t* order_host, int64_t len);

/* The same order evaluated by the device kernel that the fused calls use, written to
 * `order_dev` (device pointer, len int32) on `stream`. */
dt_status dt_swizzle_plan_device(const dt_args* a, int op, int32_t* order_dev, int64_t len,
                                 void* stream);

/* Synchronise `stream`, read and clear the workspace's device error word.
 * Returns DT_OK or DT_ERR_TIMEOUT; `info` (may be NULL) receives 4 words:
 * {device code, site, detail0, detail1}. */
dt_status dt_check(void* workspace, void* stream, uint32_t* info);

/* Bytes of the fixed device scratch behind dt_ag_gemm_static_scratch. */
#define DT_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* Fused AllGather-GEMM for callers that cannot allocate device memory: a plugin whose host
 * framework owns all device memory and gives it no workspace, a process that reserved the
 * whole GPU for its own allocator, or a latency-critical path that cannot afford
 * cudaMalloc's device-wide synchronisation.  Same arguments and results as dt_ag_gemm
 * without the workspace: the scratch is a fixed DT_STATIC_SCRATCH_BYTES device array inside
 * the library, which every GPU that loads the library holds until the process exits.
 *   - Problems with dt_workspace_size(a, DT_OP_AG_GEMM) > DT_STATIC_SCRATCH_BYTES are
 *     rejected with DT_ERR_WORKSPACE; argument errors as in dt_ag_gemm.
 *   - Transfer backends: DT_XFER_TMA or DT_XFER_LDST (DT_XFER_AUTO means TMA); the copy
 *     engine needs a side stream and returns DT_ERR_UNSUPPORTED.
 *   - Allocates nothing: no cudaMalloc / cudaFree, no stream or event creation.
 *   - The first call on each device resolves the array's device address (once per device,
 *     with that device current); make that first call before any stream capture begins.
 *   - All calls on a device share the one array and it keeps the last call's contents; each
 *     call clears its error word and layout tag first, so the tile order, flags and counters
 *     are rebuilt every call.  Calls that overlap on the GPU race: order them.
 *   - Bounded device waits still end a stalled call; the error they record stays in the
 *     array until dt_static_scratch_check() reads it (the next call clears it first).
 * The pages have no counterpart of this entry point. */
dt_status dt_ag_gemm_static_scratch(const void* const* a_shards, const void* b, void* c,
                                    const dt_args* a, void* stream);

/* dt_check() for the fixed scratch of the current device: synchronise `stream`, read and clear
 * the error block that the last dt_ag_gemm_static_scratch call on this device left in the
 * array.  Returns DT_OK, DT_ERR_TIMEOUT (a bounded device wait ran out: C is incomplete) or
 * DT_ERR_INVALID; `info` (may be NULL) receives {device code, site, detail0, detail1}.
 * Allocates nothing.  Call it after the static-scratch call it checks and before the next one. */
dt_status dt_static_scratch_check(void* stream, uint32_t* info);

/* One candidate of the tuner: its knobs, mean time per call (ms, < 0 if it did not run) and
 * the status of its calls. */
typedef struct dt_tune_point {
  int64_t chunk_rows;
  int32_t backend;    /* dt_xfer as requested (AllGather)       */
  int32_t copy_ctas;
  int32_t swizzle;
  int32_t group;
  int32_t tile_m;     /* tile rows as requested (0 = the library's choice) */
  int32_t col_band;   /* column band as requested (0 = automatic) */
  float ms;
  int32_t status;     /* dt_status of the candidate's calls      */
} dt_tune_point;

/* sizeof(dt_tune_point) as compiled into the library, for bindings to check their mirror. */
size_t dt_sizeof_tune_point(void);

/* Enumerate-and-measure tuner (AutoOverlap page, section 6: the inter-chunk tuner picks chunk
 * size / split factor, the intra-chunk tuner the transfer backend, the SMs given to
 * communication and the tile order, all by measuring the generated variants).
 * AllGather-GEMM candidates: chunk rows {64 .. 4096, M/W} x {copy engine (when the chunk count
 * stays <= 512), TMA and ld/st with co-located transfer warps, TMA and ld/st on 8 or 16
 * dedicated CTAs, the per-tile pull DT_XFER_TMA_TILE when (M/W) % 128 == 0} x column bands
 * {as given, one band} when the given (or automatic) bands are more than one; then group
 * widths {4, 8, 16} at the best point.  Scatter-mode candidates
 * (dt_tune_reduce with op DT_OP_GEMM_RS, DT_OP_GEMM_AR or DT_OP_GEMM_A2A): chunk rows x group
 * widths {4, 8, 16}, at the tile rows given, and for DT_OP_GEMM_RS / DT_OP_GEMM_AR x column
 * bands {as given, one band} when the given (or automatic) bands are more than one.  A
 * candidate whose group width or column band gives the same tile order as an earlier one with
 * the same chunk rows, tile rows and transfer is not timed.  Each candidate runs once as
 * warm-up and `reps` times timed with CUDA events on `stream` (synchronising).  A forward
 * pass times every candidate and takes the fastest as the reference; a reverse pass times each
 * other candidate between two timings of the reference and scores it by its time over their
 * mean (the GPU's clock drifts as it warms under the power cap; the ratio cancels the drift);
 * a point's reported ms is its score times the reference's median time.  Candidates whose
 * workspace exceeds ws_bytes are skipped.  The knobs kept are those that move the fewest DRAM
 * bytes among near-equal points (a short timing at full clock does not show DRAM bytes, a run
 * under the power cap does): for the reduce ops the automatic column bands unless one band is
 * more than 4 % faster, then, among the points of the kept band setting within 1 % of its
 * fastest, the largest chunk rows, then the fastest; for the AllGather, among the points within
 * 1 % of the fastest, the largest chunk rows (fewer key groups re-stream B fewer times), then
 * the fastest.  They are written into *a (chunk_rows, backend, copy_ctas, group, tile_m, col_band;
 * swizzle stays on).  `points` (may be NULL) receives
 * up to max_points candidates and *n_points their number.  The inputs are read and the
 * outputs written by every candidate; all candidates give bit-identical outputs. */
dt_status dt_tune_ag_gemm(const void* const* a_shards, const void* b, void* c, void* workspace,
                          size_t ws_bytes, dt_args* a, int32_t reps, dt_tune_point* points,
                          int32_t max_points, int32_t* n_points, void* stream);
dt_status dt_tune_reduce(int op, const void* const* a, const void* const* b, void* const* out,
                         void* workspace, size_t ws_bytes, dt_args* a_args, int32_t reps,
                         dt_tune_point* points, int32_t max_points, int32_t* n_points,
                         void* stream);

/* Environment settings, read once per process at the first call that needs them (for
 * measurement and comparison; the defaults are the library's choices):
 *   DT_PDL=0        launch the fused kernel without programmatic stream serialization (default 1:
 *                   its launch and set-up overlap the prepare kernel before it; it waits for that
 *                   grid before it touches global memory).
 *   DT_RS_REDUCE=0  ReduceScatter / AllReduce middle sources fold with a load, an add and a store
 *                   (default 1: a TMA reduce-add into the running sum; same bits).
 *   DT_ROT=r        ReduceScatter / AllReduce: the CTA pairs' slot in each wave of the tile order
 *                   rotates by r per wave (default 1; 0: the same slot every wave; same bits).
 *   DT_L2_HINTS=h   ReduceScatter / AllReduce L2 policies: bit 0 running sums, park slots and
 *                   final sums evict first, bit 1 B_q evict last (default 3).
 *   DT_C_TMA=0      AllGather-GEMM / AllToAll outputs stored per thread (default 1: TMA stores).
 *   DT_COPY_PIECE=b, DT_COPY_BUFS=n   dedicated in-kernel transfer workers' piece size (8192,
 *                   16384 or 32768 bytes; default 32768) and buffers per worker (1-4; default 1).
 * Every setting gives the same output bits. */

/* Failure-detection testing, host side only: the next AllGather-GEMM call on this process
 * (dt_ag_gemm on any backend, or dt_ag_gemm_static_scratch) leaves out the copy and the
 * ready-flag write of transfer step `step` (the position in the gather order; -1 clears): the
 * copy engine is not given that copy, or the in-kernel transfer is told to skip that chunk.
 * The tiles that need that chunk wait until `timeout_us`, record DT_ERR_TIMEOUT in the
 * workspace (or the fixed scratch) and exit; the CUDA context stays usable.  (Syncopate summary page, "局限与后续工作": fault injection for lost signals and
 * timeouts.) */
dt_status dt_debug_drop_transfer(int32_t step);

/* Debug timeline of the fused AllGather-GEMM: how much of the chunk transfer the GEMM hid.
 * (DITRON page, paper section 4.1: most of the communication of a large AllGather-GEMM is
 * hidden behind the GEMM; AutoOverlap page, section 2: what kernel-level overlap leaves
 * exposed.)  While a buffer is attached, every dt_ag_gemm call (and every dt_allgather call on
 * an in-kernel backend, whose kernel has no GEMM: words [2], [3] and [6 + 3c] stay as reset)
 * resets it on its stream and its kernel records, in 64-bit global-timer nanoseconds:
 *   [0] first CTA start, [1] last CTA exit, [2] total time the GEMM's producers spent waiting
 *   for ready flags (summed over waits), [3] how many waits found their chunk missing;
 *   then per chunk c = s * nC + j (rank s, chunk j):
 *   [4 + 3c] release of its ready flag by the in-kernel transfer (all ones on the copy engine,
 *            whose stream writes the flag), [5 + 3c] the first wait that found it missing
 *            began (all ones if none did), [6 + 3c] the first tile read past its flag (all ones
 *            for chunks read in place or never waited for).
 * `trace` is caller-owned device memory of at least dt_trace_bytes(a) bytes, 8-byte aligned;
 * NULL detaches.  A call whose problem needs more bytes than attached returns DT_ERR_INVALID.
 * Tracing adds a few global atomics per chunk and per CTA; it is off unless attached. */
size_t dt_trace_bytes(const dt_args* a);
dt_status dt_trace_attach(void* trace, size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* DT_H_ */
