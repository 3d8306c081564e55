/*
 * attn.h — C ABI of the GB300 (sm_103a) attention-forward library.
 *
 * One call computes, for every batch b, query head h and query row i,
 *
 *   O[b,h,i,:] = softmax_j( scale * Q[b,h,i,:] . K[b,kvh,j,:] ) V[b,kvh,j,:]
 *
 * over the keys j that are visible to row i, plus the row's log-sum-exp.
 * Sources (web pages this library restates):
 *   - "Flash Attention in CUDA Tile (cuTile)" (NVIDIA blog), sections
 *     "What is attention?" and "Understanding online softmax": the operation
 *     and the tiled online-softmax method that computes it exactly;
 *   - same page, section "Causal attention" and the kernel listing's
 *     "Applying the causal mask" step: key j is visible to query row i iff
 *     j <= input_pos + i (queries sit at absolute positions input_pos + i,
 *     the KV-cache offset of the listing's "Initializing accumulators" step);
 *   - same page, section "Grouped-query attention": kvh = h / (Hq / Hkv);
 *   - same page, host-launcher section: [B, H, S, D] contiguous tensors,
 *     the scale defaulting to 1/sqrt(D) on the Python side.
 *
 * No function here allocates device memory; the caller owns every buffer.
 * (attn_fwd_splitkv_noalloc's scratch is a fixed array compiled into the
 * library, which every GPU that loads it holds, not an allocation.)
 */
#ifndef ATTN_FWD_GB300_ATTN_H
#define ATTN_FWD_GB300_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
struct CUstream_st;
typedef struct CUstream_st* attn_stream_t;

/* Element type of Q, K, V and O. */
typedef enum {
  ATTN_F16 = 0,  /* IEEE binary16 */
  ATTN_BF16 = 1, /* bfloat16 */
  ATTN_E4M3 = 2  /* OCP FP8 E4M3 ("e4m3fn") inputs with a bfloat16 O: only
                    attn_fwd_fp8, attn_splitkv_plan and attn_tile_config
                    take it; elsewhere ATTN_ERR_INVALID_ARG (ATTN_ERR_-
                    UNSUPPORTED for attn_bwd) */
} attn_dtype_t;

/* Return codes.  Everything but ATTN_OK leaves O and LSE untouched. */
typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* bad size, NULL or host pointer, bad dtype   */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (D not 64 or 128) */
  ATTN_ERR_ALIGNMENT = 3,    /* Q/K/V/O not 16-byte or LSE not 4-byte aligned */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed            */
  ATTN_ERR_TIMEOUT = 5       /* a kernel pipeline wait ran out (device status) */
} attn_status_t;

/*
 * attn_fwd — scaled-dot-product attention forward on the GPU.
 *
 * Q    device, [B, Hq,  Sq,  D] contiguous, dtype      (read)
 * K    device, [B, Hkv, Skv, D] contiguous, dtype      (read)
 * V    device, [B, Hkv, Skv, D] contiguous, dtype      (read)
 * O    device, [B, Hq,  Sq,  D] contiguous, dtype      (written)
 * LSE  device, [B, Hq,  Sq] float32, or NULL to skip   (written)
 *      LSE[b,h,i] = ln( sum over visible j of exp(scale * q_i . k_j) ),
 *      natural log, scale included.
 * B >= 0, Hq > 0, Hkv > 0 with Hq % Hkv == 0, Sq >= 0, Skv >= 1,
 * D in {64, 128}.  B == 0 or Sq == 0 is a successful no-op.
 * scale     finite; any sign (0 gives uniform weights over visible keys).
 * causal    0: every key is visible and input_pos is ignored;
 *           non-zero: key j is visible to query row i iff j <= input_pos + i.
 *           Queries with input_pos + i >= Skv - 1 see every key.
 * input_pos >= 0, and input_pos + Sq + 512 must fit in a signed 32-bit int.
 * dtype     ATTN_F16 or ATTN_BF16 (Q, K, V and O share it).
 * stream    the CUDA stream the kernel is enqueued on.
 *
 * Q/K/V/O must be 16-byte aligned (tensor-memory-accelerator copies), LSE
 * 4-byte aligned; O must not overlap Q, K or V.  The call is asynchronous:
 * the return code covers argument checks and the launch only.  A device
 * side pipeline timeout is reported later by attn_device_status().
 * Results are deterministic for a given shape and dtype.
 */
attn_status_t attn_fwd(const void* Q, const void* K, const void* V, void* O,
                       float* LSE, int B, int Hq, int Hkv, int Sq, int Skv,
                       int D, float scale, int causal, int input_pos,
                       attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_fwd_window — attn_fwd with a causal sliding window: the query at
 * absolute position p = input_pos + i sees the keys j with
 * p - window < j <= p (its last `window` positions, itself included).
 * "Flash Attention from Scratch", section "What's Next", names sliding
 * window attention for ultra-long sequences as future work without
 * defining it; this is the plain reading consistent with the causal offset
 * rule above.  Key tiles wholly before a query tile's window are skipped
 * like those past its causal horizon.
 *
 * Arguments as attn_fwd, plus:
 * window   >= 0 keys; 0 means no window (the result of attn_fwd).  A
 *          window needs causal != 0, and every query must see a key
 *          (input_pos + Sq - window < Skv); otherwise
 *          ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_fwd_window(const void* Q, const void* K, const void* V,
                              void* O, float* LSE, int B, int Hq, int Hkv,
                              int Sq, int Skv, int D, float scale, int causal,
                              int input_pos, int window, attn_dtype_t dtype,
                              attn_stream_t stream);

/*
 * attn_fwd_splitkv — the same operation as attn_fwd, with the key range cut
 * into num_splits pieces of equal length (multiples of 128 keys) that are
 * processed in parallel, then merged by their log-sum-exps: for a row with
 * partial results (O_c, lse_c), O = sum_c w_c O_c / sum_c w_c and
 * LSE = M + ln(sum_c w_c) with w_c = exp(lse_c - M), M = max_c lse_c.
 * This is the KV-cache decoding shape (few query rows, long key range)
 * where attn_fwd alone would leave most SMs idle; it is the online-softmax
 * rescaling of "Flash Attention in CUDA Tile (cuTile)", section "The online
 * softmax algorithm", applied across key ranges.
 *
 * Arguments as attn_fwd, plus:
 * num_splits       1..128, a value returned by attn_splitkv_plan for the
 *                  same shape (other counts give ATTN_ERR_INVALID_ARG);
 * workspace        device memory owned by the caller, 256-byte aligned,
 *                  of at least the size attn_splitkv_plan reports: fp32
 *                  partial outputs [num_splits, B, Hq, Sq, D], fp32
 *                  partial LSEs [num_splits, B, Hq, Sq]; its contents
 *                  need no initialisation (every value read is written
 *                  first by the same call);
 * workspace_bytes  its size.
 * Enqueued on `stream`: the forward kernel, and unless its key ranges merge
 * inside thread-block clusters (GQA-packed launches whose units all run at
 * once, at most 8 ranges), a merge kernel after it (a programmatic
 * dependent launch: its blocks start once every forward block has and wait
 * for the forward grid to complete).  The workspace must not be used by
 * another call until this one has run.
 */
attn_status_t attn_fwd_splitkv(const void* Q, const void* K, const void* V,
                               void* O, float* LSE, int B, int Hq, int Hkv,
                               int Sq, int Skv, int D, float scale, int causal,
                               int input_pos, attn_dtype_t dtype,
                               int num_splits, void* workspace,
                               size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_fwd_splitkv_window — attn_fwd_splitkv with the sliding window of
 * attn_fwd_window (same `window` rule).  Plan with attn_splitkv_plan (the
 * plan does not depend on the window); ranges wholly outside a row
 * block's window are skipped.
 */
attn_status_t attn_fwd_splitkv_window(const void* Q, const void* K,
                                      const void* V, void* O, float* LSE,
                                      int B, int Hq, int Hkv, int Sq, int Skv,
                                      int D, float scale, int causal,
                                      int input_pos, int window,
                                      attn_dtype_t dtype, int num_splits,
                                      void* workspace, size_t workspace_bytes,
                                      attn_stream_t stream);

/*
 * attn_fwd_fp8 — attention forward with 8-bit floating-point inputs.
 * "Flash Attention from Scratch", section "What's Next", names FP8 tensor
 * cores as future work without defining a format; the reading taken: Q, K
 * and V hold OCP E4M3 codes (sign, 4-bit exponent with bias 7, 3-bit
 * mantissa, no infinities, S.1111.111 is NaN; torch.float8_e4m3fn) with one
 * fp32 descale factor per tensor, and the call computes the operation of
 * attn_fwd_window on the real values
 *   Q = q_descale * Q8,  K = k_descale * K8,  V = v_descale * V8.
 * Both products run on the FP8 tensor cores with fp32 accumulation; the
 * softmax weights are rounded to E4M3 for the P.V product (the row sums
 * use them unrounded), which bounds the accuracy: each weight carries up to
 * 2^-4 relative rounding (absolute 2^-10 below 2^-6).  The LSE is exact to
 * fp32 rounding.
 *
 * Q, K, V  device, layouts as attn_fwd, one byte per element (read);
 * O        device, [B, Hq, Sq, D] bfloat16 (written);
 * LSE      device fp32 [B, Hq, Sq] or NULL: ln-sum-exp of the scores
 *          scale * q_descale * k_descale * Q8.K8 (written);
 * D        128 only (else ATTN_ERR_UNSUPPORTED);
 * scale, q_descale, k_descale, v_descale  finite, any sign; the product
 *          scale * q_descale * k_descale must be finite in fp32;
 * causal, input_pos, window  as attn_fwd_window;
 * num_splits  0: one pass (workspace ignored); >= 1: the split-KV form of
 *          attn_fwd_splitkv_window with a count from attn_splitkv_plan
 *          (dtype ATTN_E4M3) and its workspace rules;
 * Other rules and errors as attn_fwd.
 */
attn_status_t attn_fwd_fp8(const void* Q, const void* K, const void* V,
                           void* O, float* LSE, int B, int Hq, int Hkv,
                           int Sq, int Skv, int D, float scale,
                           float q_descale, float k_descale, float v_descale,
                           int causal, int input_pos, int window,
                           int num_splits, void* workspace,
                           size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_splitkv_plan — split count and workspace size for attn_fwd_splitkv.
 * *num_splits in: the requested count, or <= 0 to choose the count with
 * the shortest estimated time on the current device's SMs (152, a GB300's,
 * when the calling thread has no CUDA device): waves of units times key
 * tiles per range plus fixed per-unit and merge costs, bounded below by
 * streaming K and V once from HBM; out: the count attn_fwd_splitkv accepts
 * (requests are clamped to the number of 128-key tiles, and trailing empty
 * ranges are dropped).  Host only: launches nothing.
 * *workspace_bytes (may be NULL) receives the workspace size.
 */
attn_status_t attn_splitkv_plan(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                int causal, int input_pos, attn_dtype_t dtype,
                                int* num_splits, size_t* workspace_bytes);

/*
 * attn_fwd_splitkv_noalloc — attn_fwd_splitkv for callers that cannot
 * allocate device memory (code running where the allocator must not be
 * entered, or inside a host that owns every allocation): the partial
 * results go to a fixed scratch array compiled into this library (its size
 * is attn_noalloc_scratch_bytes(), 16 MiB, held on every GPU that loads the
 * library until the process exits) instead of a caller workspace.  The
 * pages have no counterpart; this is a deployment convenience.
 *
 * Arguments as attn_fwd_splitkv without the workspace: num_splits <= 0
 * lets the library choose, and a positive count must be one that
 * attn_splitkv_plan keeps (otherwise ATTN_ERR_INVALID_ARG).  Returns
 * ATTN_ERR_UNSUPPORTED when the partial results of that split count need
 * more than the scratch holds.  The first call on a device (and the first
 * after a device reset, which replaces the context) looks up the scratch
 * address on that device (no allocation); make that first call before any
 * stream capture.  All calls share the one scratch array and it keeps the
 * last call's contents (nothing in it has to start at zero): calls whose
 * kernels overlap on the GPU race on it, so issue them on one stream or
 * otherwise order them.
 */
attn_status_t attn_fwd_splitkv_noalloc(const void* Q, const void* K,
                                       const void* V, void* O, float* LSE,
                                       int B, int Hq, int Hkv, int Sq, int Skv,
                                       int D, float scale, int causal,
                                       int input_pos, attn_dtype_t dtype,
                                       int num_splits, attn_stream_t stream);

/* Bytes of the fixed scratch array attn_fwd_splitkv_noalloc uses. */
size_t attn_noalloc_scratch_bytes(void);

/*
 * attn_bwd — backward pass: gradients dQ, dK, dV of the forward output O
 * for an upstream gradient dO.  "Flash Attention from Scratch", section
 * "What's Next", lists the backward pass as future work without formulas;
 * this is the chain rule on the forward's definition, recomputing P tile
 * by tile from the forward's LSE instead of storing it:
 *   P_ij = exp(scale q_i.k_j - LSE_i) on visible keys (0 elsewhere),
 *   D_i = sum_d dO_id O_id,  dV_j = sum_i P_ij dO_i,
 *   dS_ij = P_ij (dO_i.v_j - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 * with the query heads of a GQA group adding into the same dK, dV.
 *
 * Q, K, V, O, dO   device, same dtype and layouts as attn_fwd (O and LSE
 *                  are the forward's outputs for these Q, K, V and scale,
 *                  causal, input_pos, window);
 * LSE              device fp32 [B, Hq, Sq] (required);
 * dQ               device [B, Hq, Sq, D]; dK, dV device [B, Hkv, Skv, D];
 *                  outputs, same dtype, 16-byte aligned, overlapping no
 *                  input, each other or the workspace;
 * window           as attn_fwd_window (0: none);
 * workspace        device, 256-byte aligned, at least
 *                  attn_bwd_workspace_bytes(B, Hq, Sq) bytes (per-row
 *                  lse2 and D); contents need no initialisation;
 * Three kernels: the row pass and the dK/dV kernel on `stream`, the dQ
 * kernel on an internal stream forked from `stream` after the row pass and
 * joined back into it (event record / wait), so the two run concurrently
 * and later work on `stream` waits for both; this works under stream
 * capture.  The first call on a host thread and device creates that
 * internal stream and its two events (make it before any capture).  Every
 * output element has one writer, so results are deterministic.  Sq = 0
 * writes zero dK, dV.  Errors as attn_fwd.
 */
attn_status_t attn_bwd(const void* Q, const void* K, const void* V,
                       const void* O, const float* LSE, const void* dO,
                       void* dQ, void* dK, void* dV, int B, int Hq, int Hkv,
                       int Sq, int Skv, int D, float scale, int causal,
                       int input_pos, int window, attn_dtype_t dtype,
                       void* workspace, size_t workspace_bytes,
                       attn_stream_t stream);

/* Workspace bytes attn_bwd needs for B x Hq x Sq query rows: two fp32
 * values per row, Sq padded to a multiple of 128 (0 on negative sizes). */
size_t attn_bwd_workspace_bytes(int B, int Hq, int Sq);

/* Short English description of a status code (static storage). */
const char* attn_status_string(attn_status_t status);

/*
 * attn_device_status — synchronises the current device, then reads and
 * clears the library's device status word.  *code receives 0 when no kernel
 * wait has run out since the last call; otherwise a non-zero code
 * (bits 0-7: 1 = wait timed out; bits 8-15: the pipeline role that gave
 * up) and the function returns ATTN_ERR_TIMEOUT.  code may be NULL.
 * Every wait of every kernel in flight ORs into the one word, so the
 * device-wide form sees them all; attn_stream_status below waits for one
 * stream only.
 */
attn_status_t attn_device_status(unsigned int* code);

/*
 * attn_stream_status — the same query ordered on one stream: waits for the
 * work already enqueued on `stream` (cudaStreamSynchronize of that stream
 * only; other streams keep running), reads the status word and enqueues on
 * `stream` the clearing of exactly the bits it reports.  The word is one
 * per device, shared by every stream and call, so a wait that ran out in a
 * kernel of another stream, finished before the read, is reported here too;
 * bits 8-15 name the role that gave up (in the forward kernel 1 producer,
 * 2 MMA issuer, 3 softmax, 4 epilogue; OR-ed when several gave up).  Not for use while `stream` is being captured.  code
 * may be NULL.
 */
attn_status_t attn_stream_status(attn_stream_t stream, unsigned int* code);

/*
 * attn_selftest_wait_timeout — exercises the kernel's bounded-wait abort
 * path on demand.  Launches the attn_fwd kernel for these arguments (same
 * meaning and checks as attn_fwd) with two changes: every pipeline wait
 * gives up after timeout_ns (> 0) instead of the library default, and the
 * first CTA never loads its first K tile, so its MMA issuer waits for a
 * tile that cannot arrive.  That wait runs out, the CTA's roles stop,
 * drain what they have in flight (bounded), free TMEM and exit; the other
 * CTAs finish normally.  Nothing faults or hangs and the context stays
 * usable: the timeout is reported by the next attn_device_status() or
 * attn_stream_status() (ATTN_ERR_TIMEOUT, bit 0 set, role bits non-zero),
 * and the rows of the first CTA's work units in O and LSE are left
 * undefined.  For tests of the failure path only.
 */
attn_status_t attn_selftest_wait_timeout(const void* Q, const void* K,
                                         const void* V, void* O, float* LSE,
                                         int B, int Hq, int Hkv, int Sq,
                                         int Skv, int D, float scale,
                                         int causal, int input_pos,
                                         attn_dtype_t dtype,
                                         unsigned long long timeout_ns,
                                         attn_stream_t stream);

/*
 * attn_tile_config — the tile configuration attn_fwd would launch for these
 * arguments (host only, no GPU needed).  Fills, when non-NULL:
 *   block_m   query rows per CTA, block_n keys per K/V tile,
 *   stages    K/V tiles the shared-memory ring holds,
 *   grid      work units (each 2 x 128 query rows); the launch runs
 *             min(grid, SM count) persistent CTAs that walk them,
 *   smem_bytes dynamic shared memory per CTA.
 * Returns the same validation code attn_fwd would (pointers not checked).
 */
attn_status_t attn_tile_config(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                               int causal, int input_pos, attn_dtype_t dtype,
                               int* block_m, int* block_n, int* stages,
                               int* grid, int* smem_bytes);

/*
 * attn_dispatch_t / attn_dispatch — the forward dispatch-table entry a call
 * with these arguments runs, spelled out (host only, no GPU needed).  The
 * entry is keyed on D, dtype, causal / window, the GQA group size and Sq
 * (the tile shape and work unit) and on num_splits (one pass or split-KV):
 *   q_tiles 2, paired 1   two query heads of one K/V group at the same 128
 *                         rows per unit (even group size);
 *   q_tiles 2, paired 0   256 consecutive rows of one head per unit;
 *   q_tiles 1             the group * Sq <= 128 query rows of all heads of
 *                         a K/V group packed into one tile (few query rows);
 *   s_buffers             score tiles in TMEM: 2, or 3 rotating between the
 *                         two Q tiles at D = 64 (O needs only 128 columns);
 *   order 0               heaviest causal row block first, the heads of a
 *                         row block in turn (longest-processing-time order
 *                         over the persistent CTAs); order 1: the row blocks
 *                         of one head in turn (non-causal: equal units, K/V
 *                         of the few heads in flight stays in L2); order 2:
 *                         causal units assigned to the CTAs by a plan packed
 *                         on the host (one-pass launches of more units than
 *                         SMs and at most 1024, when the plan beats the
 *                         order-0 rounds; see attn_unit_plan), so the entry
 *                         depends on Sq through the unit count;
 *   o_store 1             O leaves through a 128-byte-swizzled shared-memory
 *                         box stored by TMA; 0: each softmax thread stores
 *                         its row (packed tiles, split-KV fp32 partials);
 *   hold_scores 1         the softmax keeps a row's 128 scores in registers
 *                         between its max and exp passes (register split).
 * units is the number of work units (the launch runs min(units, SM count)
 * persistent CTAs), stages the K/V tiles in flight, smem_bytes the dynamic
 * shared memory per CTA.  name is a static string naming the entry.
 * num_splits: 0 for the one-pass forward, else as attn_fwd_splitkv
 * (planned count; units then count (rows, key range) pairs).  merge: how
 * the key ranges are merged -- 0 no split; 1 inside the forward kernel,
 * the ranges of a K/V group forming one thread-block cluster (packed tiles,
 * units <= SM count, at most 8 ranges; one kernel per call); 2 by a merge
 * kernel enqueued after the forward kernel (two kernels per call).  The
 * SM count is the current device's (152 without one).  Returns the
 * validation code the call would; out must be non-NULL.
 */
typedef struct {
  int block_m, block_n, q_tiles, paired, s_buffers, stages;
  int order, o_store, hold_scores, num_splits, units, smem_bytes, merge;
  const char* name;
} attn_dispatch_t;

attn_status_t attn_dispatch(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                            int causal, int input_pos, int window,
                            attn_dtype_t dtype, int num_splits,
                            attn_dispatch_t* out);

/*
 * attn_unit_plan — how a one-pass forward call of this shape assigns its
 * work units to `grid` persistent CTAs (host only, no GPU needed; the call
 * itself uses grid = min(units, SM count)).  Has no counterpart in the
 * method's description: it exposes the launch's load balancing.
 * Causal two-tile launches (not the packed few-row mode) of more units
 * than CTAs and at most 1024 units are packed on the host: units heaviest
 * first into the first CTA with room under a capacity searched from the
 * mean upwards (first-fit decreasing, the MULTIFIT method), kept only when
 * its busiest CTA beats the zigzag rounds the kernel otherwise walks.
 *   planned      out: 1 when such a plan assigns the units, else 0 (the
 *                rounds: non-causal or packed launches, units <= grid,
 *                more than 1024 units, or no better plan);
 *   work_max     out: the busiest CTA's work under the assignment the
 *                call uses, in half K/V steps (each unit counts 2 per K/V
 *                step its later Q tile visits, plus 3 for its boundary);
 *                0 when not computed (a launch the plan never considers);
 *   work_rounds  out: the same under the zigzag rounds (0 likewise);
 *   unit_order   optional (NULL: not written), room for the unit count:
 *                CTA c walks units unit_order[cta_start[c] ..
 *                cta_start[c + 1]) in order (written only when planned);
 *   cta_start    optional, room for min(units, grid) + 1 entries.
 * Returns the validation code of attn_fwd for the shape (bf16), or
 * ATTN_ERR_INVALID_ARG for grid < 1 or a NULL output.
 */
attn_status_t attn_unit_plan(int B, int Hq, int Hkv, int Sq, int Skv, int D,
                             int causal, int input_pos, int window, int grid,
                             int* planned, long long* work_max,
                             long long* work_rounds, int* unit_order,
                             int* cta_start);

/* Library version as major*10000 + minor*100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_GB300_ATTN_H */
