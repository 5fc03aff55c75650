/*
 * tide.h — C ABI of the GB300 (sm_103a) layout-aware reduce-scatter and all-gather placement.
 *
 * "TIDE" is the paper "The Endgame of FSDP Communication: Layout-Aware Collectives on Copy
 * Engines, RDMA, and NVSwitch" (arXiv 2610.38228).  Citations below name its abstract, figures
 * and tables.
 *
 * Model.  An FSDP2 parameter group holds P parameters; parameter p has rows_p rows (dim 0) of
 * row_len_p = L_p elements (the product of its other dims; 1 for a 1-D tensor), row-major and
 * contiguous.  It is sharded on dim 0 over R ranks (abstract; Fig. 1):
 *     m_p = ceil(rows_p / R)                    padded rows per rank         (Table 2)
 *     s_p = m_p * L_p                           per-rank shard elements      (Table 2)
 *     o_p = s_0 + ... + s_{p-1}                 prefix offset in a shard     (Table 2)
 *     S   = sum_p s_p,   U = sum_p rows_p*L_p   packed shard / unsharded     (Table 2)
 *     v(d,p) = clamp(rows_p - d*m_p, 0, m_p)    valid rows of p on rank d (the rest is padding)
 * Rank d's piece of p is the contiguous element range [d*s_p, d*s_p + v(d,p)*L_p) of the tensor,
 * and it lives at elements [o_p, o_p + s_p) of rank d's packed shard, padding rows last.
 * On one GPU the R ranks are R separate buffers in that GPU's memory.
 *
 * Conventions for every call:
 *   - All sizes and offsets are elements (int64).  Returns TIDE_OK (0) or a negative status.
 *   - Device pointers are plain CUDA device addresses on the device that was current when the
 *     group was created; that device must be current at every call on the group.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).  Collective
 *     calls are asynchronous and stream-ordered: they return once the work is enqueued.  Their
 *     inputs must stay alive and unmodified, and their outputs untouched, until the stream has
 *     executed the call.  Errors raised by the kernels themselves surface at the next
 *     synchronisation of that stream; argument errors are returned before anything is enqueued.
 *   - Host pointer arrays (grads, shards, params, slots) are copied before the call returns.
 *   - The caller owns every device buffer.  A group owns only its plan tables (device), a small
 *     ring of pinned host / device pointer tables and CUDA events; tide_group_destroy frees them.
 *   - A group may be used from several host threads; calls on one group are serialised.
 *   - Inputs and outputs of one call must not overlap.  Nothing here traps on the device.
 */
#ifndef TIDE_H
#define TIDE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------------ */
#define TIDE_OK 0
#define TIDE_EINVAL (-1)  /* null pointer, R < 1, P < 1, rows < 1, row_len < 1, bad index, wrong device,
                            or a device pointer not aligned to its element (2 bytes bf16, 4 bytes fp32) */
#define TIDE_EALIGN (-2)  /* TIDE_FLAG_VEC_STRICT set and a pointer that needs 16-byte alignment lacks it
                            (reduce-scatter: a gradient or a staging slot; placement: a shard or a
                            parameter) */
#define TIDE_ELAYOUT (-3) /* TIDE_FLAG_CE_STRICT set and the shards are not at a uniform pitch */
#define TIDE_ECUDA (-4)   /* a CUDA runtime call failed; tide_last_cuda_error() gives its code */
#define TIDE_ENOMEM (-5)  /* host or device allocation of the group's own tables failed */
#define TIDE_ERANGE (-6)  /* a size overflows int64, or R*P exceeds TIDE_MAX_TABLE */

#define TIDE_MAX_RANKS 4096
#define TIDE_MAX_TABLE (1 << 22) /* max R*P pointer-table entries */

/* ---- group flags ------------------------------------------------------------------------- */
/* Return TIDE_EALIGN instead of running the element-wise path when a pointer whose 16-byte
 * alignment the vector paths need is not 16-byte aligned: a gradient for tide_reduce_scatter, a
 * staging slot for tide_reduce_scatter_slots, a shard or a parameter for tide_all_gather. */
#define TIDE_FLAG_VEC_STRICT 0x1u
/* With TIDE_FLAG_CE_2D: return TIDE_ELAYOUT from tide_all_gather_ce instead of falling back to
 * 1-D copies when shards[r] != shards[0] + r*pitch for one pitch >= S*2 bytes. */
#define TIDE_FLAG_CE_STRICT 0x2u
/* tide_all_gather_ce always issues one 2-D copy per parameter (the paper's form, about P copies;
 * see tide_group_set_ce_bands) when the shards sit at a uniform pitch. */
#define TIDE_FLAG_CE_2D 0x4u
/*
 * Interference-first defaults, for collectives that run beside compute (Fig. 3, Fig. 4, Table 4):
 * both SM kernels launch about a ninth of the SMs as CTAs (16 on a 152-SM GB300) instead of filling
 * the GPU, and tide_all_gather_ce uses one copy-engine lane (its form rule unchanged).  Measured on GB300
 * beside a single-wave cuBLAS bf16 GEMM (4096 x 4096 x 8192): the GEMM slows by a few percent
 * instead of +1400 % (reduce-scatter), +290 % (SM placement) and +60 % (copy engines, 8 lanes) at
 * the throughput-first defaults, while the collectives move a quarter to two thirds as many bytes
 * per second.  Without this flag the defaults are throughput-first: every SM, eight lanes.
 * tide_group_set_ctas / tide_group_set_ce_lanes still override either default.
 */
#define TIDE_FLAG_OVERLAP 0x8u
/* tide_all_gather_ce always issues one 1-D copy per (rank, parameter) run of valid rows (R*P
 * copies at most).  Not combinable with TIDE_FLAG_CE_2D or TIDE_FLAG_CE_STRICT.  With neither
 * TIDE_FLAG_CE_1D nor TIDE_FLAG_CE_2D the form is chosen per group (see tide_all_gather_ce). */
#define TIDE_FLAG_CE_1D 0x10u

typedef struct tide_group *tide_group_t;

/* ---- planner ----------------------------------------------------------------------------- */
/*
 * tide_plan_layout — the Table 2 quantities of a group, host only (no CUDA call).
 * In:  R ranks, P parameters, rows[P] (dim 0), row_len[P] (product of the other dims).
 * Out: m[P], s[P], o[P] (caller-allocated, P entries each), *S, *U, as defined above.
 * Errors: TIDE_EINVAL (null, R < 1, R > TIDE_MAX_RANKS, P < 1, rows < 1, row_len < 1),
 *         TIDE_ERANGE (a size overflows int64).  Outputs are untouched on error.
 */
int tide_plan_layout(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                     int64_t *m, int64_t *s, int64_t *o, int64_t *S, int64_t *U);

/*
 * tide_group_create — plan a group (abstract; Fig. 1; Table 2) and upload its work tables to
 * the current device.  `flags` is a bitwise OR of TIDE_FLAG_*.  On success *out owns the plan;
 * on error *out is set to NULL.
 * Errors: as tide_plan_layout, plus TIDE_EINVAL (an unknown flag, or TIDE_FLAG_CE_1D with
 * TIDE_FLAG_CE_2D or TIDE_FLAG_CE_STRICT), TIDE_ERANGE (R*P > TIDE_MAX_TABLE), TIDE_ENOMEM,
 * TIDE_ECUDA.
 */
int tide_group_create(tide_group_t *out, int32_t R, int32_t P, const int64_t *rows,
                      const int64_t *row_len, uint32_t flags);

/* Frees the group's tables after waiting for its own work in flight.  NULL is accepted. */
int tide_group_destroy(tide_group_t g);

/* Per-rank packed shard elements S / unsharded group elements U. */
int tide_group_shard_elems(tide_group_t g, int64_t *S);
int tide_group_unsharded_elems(tide_group_t g, int64_t *U);

/* Padded per-rank rows m_p and prefix offset o_p of parameter p (0 <= p < P). */
int tide_group_param_layout(tide_group_t g, int32_t p, int64_t *m_p, int64_t *o_p);

/* Valid rows v(d,p) that rank d holds of parameter p. */
int tide_group_valid_rows(tide_group_t g, int32_t d, int32_t p, int64_t *v);

/*
 * CTA counts of the reduce-scatter and all-gather kernels.  0 restores the default: throughput-
 * first, enough CTAs to fill every SM (one per SM for the bulk-copy reduce-scatter, two for its
 * register path, four per SM for either placement kernel), or, for a group created with
 * TIDE_FLAG_OVERLAP, sm_count / 9 CTAs for both.  A positive value is used as given (at most the
 * work's chunk count), so a caller can leave SMs to concurrent compute (Fig. 3, Fig. 4, Table 4).
 */
int tide_group_set_ctas(tide_group_t g, int32_t rs_ctas, int32_t ag_ctas);
int tide_group_get_ctas(tide_group_t g, int32_t *rs_ctas, int32_t *ag_ctas);

/* ---- collectives ------------------------------------------------------------------------- */
/*
 * tide_reduce_scatter — layout-aware mixed-precision reduce-scatter (abstract: the reduce-scatter
 * takes each parameter's bf16 gradient tensor as it is and sums into fp32 shards; Table 1, the
 * in-place read row; Fig. 2b step 5).  For every destination rank d and parameter p:
 *     shard_d[o_p + i] = g_0[i'] + g_1[i'] + ... + g_{R-1}[i'],  i' = d*s_p + i,  i < v(d,p)*L_p
 *     shard_d[o_p + i] = +0.0f                                   v(d,p)*L_p <= i < s_p
 * where g_r is rank r's bf16 gradient of p, widened exactly to fp32 and added in ascending
 * rank order with IEEE fp32 round-to-nearest-even adds (no FMA, no flush-to-zero).  The
 * shards are overwritten, not accumulated into, and not averaged.
 *   grads:  host array of R*P device pointers, entry [r*P + p] = rank r's bf16 gradient of p
 *           (rows_p*L_p elements, row-major, contiguous).  Read only, never packed.
 *   shards: host array of R device pointers, entry d = rank d's fp32 shard of S elements.
 * With 16-byte aligned gradient pointers the gradients are read with 16-byte loads or bulk copies
 * (pieces whose offset d*s_p is a multiple of 8 elements) and the sums are stored with the widest
 * vectors each shard address allows (shards need only fp32 alignment); gradient pointers that are
 * not 16-byte aligned take an element-wise path with the same results (or TIDE_EALIGN under
 * TIDE_FLAG_VEC_STRICT).
 */
int tide_reduce_scatter(tide_group_t g, const void *const *grads, void *const *shards,
                        void *stream);

/*
 * tide_reduce_scatter_slots — the summing step of the same reduce-scatter when the R ranks are R
 * GPUs (Fig. 2b: GPU d pulls slice d of every contributor, then step 5 sums; Fig. 6a: the sums are
 * formed where the shard lives).  Destination rank d first receives, from every contributor r, the
 * valid elements of its slice of each parameter into a staging slot (one contiguous copy per
 * (r, p): elements [d*s_p, d*s_p + v(d,p)*L_p) of g_r,p to slot_r[o_p ..)); this call then sums the
 * R slots into d's fp32 shard:
 *     shard[o_p + i] = slot_0[o_p + i] + slot_1[o_p + i] + ... + slot_{R-1}[o_p + i],  i < v(d,p)*L_p
 *     shard[o_p + i] = +0.0f                                                    v(d,p)*L_p <= i < s_p
 * with the same widening, order and rounding as tide_reduce_scatter, so the shard has the bits of
 * tide_reduce_scatter's shard d over the gradients the slots were filled from.
 *   d:     destination rank, 0 <= d < R.
 *   slots: host array of R device pointers, entry r = the bf16 slot (S elements) holding
 *          contributor r's slice; padding positions of the slots are never read.
 *   shard: device pointer to d's fp32 shard of S elements (overwritten).
 * Runs the bulk-copy kernel with the group's reduce-scatter CTA count; slot pointers that are not
 * 16-byte aligned take its element-wise path with the same results (or TIDE_EALIGN under
 * TIDE_FLAG_VEC_STRICT).  Asynchronous on `stream`.  Errors: TIDE_EINVAL (null or misaligned
 * pointers, d out of range, another device current), TIDE_ECUDA.
 */
int tide_reduce_scatter_slots(tide_group_t g, int32_t d, const void *const *slots, void *shard, void *stream);

/*
 * tide_stage_slices — the exchange that fills destination d's staging slots for
 * tide_reduce_scatter_slots (Fig. 2b: GPU d pulls slice d of every contributor).  For every
 * contributor r, in the order d+1, ..., R-1, 0, ..., d, and every parameter p with v(d,p) > 0, one
 * cudaMemcpyAsync (copy engines; spread over the group's copy-engine lanes, stream-ordered with
 * `stream` on both sides) of elements [d*s_p, d*s_p + v(d,p)*L_p) of grads[r*P + p] to element o_p
 * of slots[r].  Padding positions of the slots are not written.
 *   grads: host array of R*P device pointers, as in tide_reduce_scatter.
 *   slots: host array of R device pointers, bf16 slots of S elements each.
 * Errors: TIDE_EINVAL (null or misaligned pointers, d out of range, another device current),
 * TIDE_ECUDA.
 */
int tide_stage_slices(tide_group_t g, int32_t d, const void *const *grads, void *const *slots, void *stream);

/*
 * tide_all_gather — all-gather placement, SM kernel (abstract: the all-gather lands each shard
 * in the parameters' own storage, with no copy-out; Fig. 1; Fig. 5b).  For every rank r and parameter p:
 *     param_p[r*s_p + i] = shard_r[o_p + i]      for i < v(r,p)*L_p
 * Padding elements of the shards are never read; nothing outside the params is written.
 *   shards: host array of R device pointers, entry r = rank r's packed bf16 shard (S elements).
 *   params: host array of P device pointers, entry p = bf16 parameter p (rows_p*L_p elements).
 */
int tide_all_gather(tide_group_t g, const void *const *shards, void *const *params,
                    void *stream);

/*
 * tide_all_gather_ce — the same placement with copy engines and no SM kernel (Table 1: the
 * all-gather takes no SM; Fig. 5b).  Two forms:
 *   - 1-D: one cudaMemcpyAsync per (rank, parameter) run of valid rows, spread over the group's
 *     copy-engine lanes (tide_group_set_ce_lanes; default 8).  Measured on GB300 this is the fast
 *     form for runs of several MB (Llama-3.1-70B layer: 6.4 TB/s), but the host spends ~2 us
 *     submitting each copy, so groups of hundreds of short runs are host-bound (Qwen3 MoE layer:
 *     3,144 copies, 0.37 TB/s).
 *   - 2-D (the paper's one strided copy per parameter), when shards[r] = shards[0] + r*pitch for
 *     one pitch >= S*2 bytes: one cudaMemcpy2DAsync over each parameter's full ranks (height
 *     f_p = floor(rows_p/m_p), width s_p*2 bytes; or one per band of ranks, see
 *     tide_group_set_ce_bands) plus at most one cudaMemcpyAsync for the rank holding its last
 *     partial piece.  ~3.5 TB/s on every workload measured, 2.6 TB/s on the Qwen3 MoE layer.
 * TIDE_FLAG_CE_1D or TIDE_FLAG_CE_2D fixes the form (TIDE_FLAG_CE_2D falls back to 1-D without a
 * uniform pitch, or returns TIDE_ELAYOUT under TIDE_FLAG_CE_STRICT).  With neither flag the group
 * takes the 2-D form when the pitch is uniform and its valid runs average less than 4 MiB, else the
 * 1-D form; the same under TIDE_FLAG_OVERLAP, over one lane (there, beside a single-wave GEMM, strided
 * copies of long runs cost far more than 1-D copies: +144 % against +6 % on the Llama-3.1-70B layer;
 * those of short runs no more: +1.8 % on the Qwen3 MoE layer, moving 4x as much).
 */
int tide_all_gather_ce(tide_group_t g, const void *const *shards, void *const *params,
                       void *stream);

/* ---- reduce-scatter kernel variants and device-side waits --------------------------------- */
#define TIDE_RS_AUTO 0     /* TIDE_RS_TMEM when every gradient pointer is 16-byte aligned, else register path */
#define TIDE_RS_REGISTER 1 /* 16-byte register loads of 8 ranks in flight per thread, 2 CTAs per SM */
#define TIDE_RS_BULK 2     /* 45 KB bulk asynchronous copies, one rank row per stage, 1 CTA per SM */
#define TIDE_RS_TMEM 3     /* the bulk path with its sums staged in Tensor Memory and stored by separate
                              writer warps (needs 16-byte aligned gradients like TIDE_RS_BULK); each CTA
                              holds its SM's whole Tensor Memory (512 columns) while it runs */

/*
 * Chooses the reduce-scatter kernel (Fig. 2b step 5 / Fig. 6a: sums formed by a bounded number of
 * CTAs fed by bulk copies), for tide_reduce_scatter and tide_reduce_scatter_slots.  All give
 * identical bits.  The bulk paths need 16-byte aligned pointers; otherwise the register path runs.
 */
int tide_group_set_rs_variant(tide_group_t g, int32_t variant);

/* The reduce-scatter kernel tide_reduce_scatter runs on g under the current settings when every
 * gradient pointer is 16-byte aligned: TIDE_RS_TMEM, TIDE_RS_BULK or TIDE_RS_REGISTER (resolves
 * TIDE_RS_AUTO). */
int tide_group_rs_kernel(tide_group_t g, int32_t *variant);

#define TIDE_AG_AUTO 0     /* bulk-copy placement when every pointer is 16-byte aligned, >= 90 % of the
                              elements lie in runs with 16-byte compatible offsets, and either the CTA
                              count is capped below the SM count or the runs average >= 1 M elements;
                              else the register path */
#define TIDE_AG_REGISTER 1 /* 16-byte register loads and stores (for runs whose shard and parameter
                              addresses differ in 16-byte alignment, 16-byte stores assembled from two
                              aligned loads each), 4 CTAs per SM */
#define TIDE_AG_BULK 2     /* 48 KB bulk copies in and out of shared memory driven by one thread per CTA */

/* Chooses the placement kernel of tide_all_gather; both write the same bits.  The bulk path needs
 * 16-byte aligned pointers; otherwise the register path runs. */
int tide_group_set_ag_variant(tide_group_t g, int32_t variant);

/* The placement kernel tide_all_gather runs on g under the current settings when every shard and
 * parameter pointer is 16-byte aligned: TIDE_AG_BULK or TIDE_AG_REGISTER (resolves TIDE_AG_AUTO). */
int tide_group_ag_kernel(tide_group_t g, int32_t *variant);

/*
 * Every device-side wait of the library's kernels (the bulk paths' mbarrier waits) gives up after
 * `timeout_ns` (0 = the default, 2 s): it writes a nonzero code to the group's device status word,
 * the CTA drains its own copies in flight and returns.  Nothing traps.
 */
int tide_group_set_wait_timeout(tide_group_t g, uint64_t timeout_ns);

/* Reads the group's device status word (0 = no wait expired; 1 = a reduce-scatter consumer wait
 * expired, 2 = a reduce-scatter producer wait expired, 4 = draining copies after an abort expired,
 * 8 = a placement load wait expired, 16 / 32 = TIDE_RS_TMEM: a consumer's wait for a drained Tensor
 * Memory buffer / a writer's wait for a filled one expired) and clears it.
 * Synchronous: copies from the device. */
int tide_group_device_status(tide_group_t g, int32_t *status);

/* Test hook: with TIDE_DEBUG_STALL_PRODUCER the bulk path's producer never signals its stages, so
 * the consumers' bounded waits expire and the status word reports it (no copy is issued). */
#define TIDE_DEBUG_STALL_PRODUCER 0x1u
int tide_group_set_debug(tide_group_t g, uint32_t flags);

/*
 * tide_stage_into_slots — Slot-Reuse staging (abstract: an optional mode that parks the gradients
 * in all-gather slots that are no longer in use; Fig. 7: the gradients are copied into a vacated slot and
 * the slot's reuse is gated on read completion).  For every rank r it copies the P gradients of
 * grads[r*P + p] with copy engines (one cudaMemcpyAsync each, stream-ordered) into slots[r], packed
 * in parameter order without padding (parameter p at element rows_0*L_0 + ... + rows_{p-1}*L_{p-1}),
 * and writes the staged addresses to staged[r*P + p] (host array of R*P pointers).  Once the copies
 * are enqueued the caller may release the gradient tensors for reuse after the stream reaches them;
 * tide_reduce_scatter(g, staged, shards, stream) then reads the slots, and the caller gates the
 * slots' next use on an event recorded after it.
 *   slot_elems: bf16 elements available in each slot (the all-gather output of the group holds
 *   R*S >= U); TIDE_ERANGE if slot_elems < U.
 */
int tide_stage_into_slots(tide_group_t g, const void *const *grads, void *const *slots, int64_t slot_elems,
                          void **staged, void *stream);

/*
 * Spreads the copy-engine work of tide_all_gather_ce and tide_stage_into_slots over `lanes`
 * (1..8, default 8) streams: the copies start after the work already enqueued on the caller's stream, and the
 * caller's stream waits for all of them, so the calls stay stream-ordered.  Several streams keep
 * several copy engines busy at once.  The helper streams are created on first use and destroyed
 * with the group.  CUDA maps streams onto CUDA_DEVICE_MAX_CONNECTIONS hardware queues (8 by
 * default); when the lanes plus the application's other busy streams exceed that, unrelated work
 * can queue behind the copies, so raise it (up to 32) before CUDA starts or use fewer lanes.
 * More lanes move more bytes but press harder on HBM and L2 beside concurrent compute (no SM is
 * taken either way); measured on GB300 with the Llama-3.1-70B layer beside a single-wave bf16
 * GEMM: 1 lane 4.5 TB/s and ~4 % GEMM slowdown, 2 lanes 6.0 TB/s and ~14 %, 8 lanes 6.4 TB/s and
 * ~60 %.  Use 1 lane when the placement overlaps compute.
 */
int tide_group_set_ce_lanes(tide_group_t g, int32_t lanes);

/*
 * Splits each parameter's 2-D copy (the uniform-pitch form of tide_all_gather_ce) into up to
 * `bands` 2-D copies over consecutive bands of ranks, spread over the copy-engine lanes like the
 * 1-D copies (1..TIDE_MAX_RANKS, default 1: the paper's single strided copy per parameter).  Measured
 * on GB300 over 8 lanes: one band per lane runs as fast as the 1-D form on long-run groups
 * (Llama-3.1-70B layer 6.45 TB/s; 8B layer 5.2 against 5.0) but slows groups of many parameters
 * (Qwen3 MoE layer: 0.39 against 2.6 TB/s with one band).
 */
int tide_group_set_ce_bands(tide_group_t g, int32_t bands);

/* Copies issued by the last tide_all_gather_ce on g, and whether the uniform-pitch form was used. */
int tide_group_last_ce_copies(tide_group_t g, int64_t *copies, int32_t *uniform_pitch);

/* ---- reduce-scatter without allocation ---------------------------------------------------- */
/* Size of the library's fixed device scratch array used by tide_reduce_scatter_noalloc. */
#define TIDE_NOALLOC_SCRATCH_BYTES (1u << 20)

/*
 * tide_reduce_scatter_noalloc — the same reduce-scatter as tide_reduce_scatter, for callers that
 * must not allocate memory.  The paper has no counterpart: it is a deployment variant of this
 * library.  tide_group_create allocates device tables and pinned host slots; a caller whose
 * framework has already reserved nearly all device memory in its own caching allocator, or that
 * cannot afford cudaMalloc/cudaFree (they may synchronise the device) while communication runs
 * beside compute, can call this instead.  It takes the group description and the pointers
 * directly (same meaning and layout as tide_group_create + tide_reduce_scatter), plans the group
 * on the host at every call into a fixed host array (no heap allocation), copies the work tables
 * into a fixed device array of TIDE_NOALLOC_SCRATCH_BYTES that the library carries (every GPU that
 * loads the library holds it until the process exits), and launches the register-path
 * reduce-scatter kernel with its default CTA count (two per SM).  It calls no cudaMalloc, cudaFree
 * or other allocating CUDA routine, and no allocating host routine either.
 *   - Size limit: the tables take round_up(56*R*P, 256) + 8*(R*P + R) bytes; a group whose
 *     tables do not fit in TIDE_NOALLOC_SCRATCH_BYTES (e.g. R = 8 with P > 2047) is rejected
 *     with TIDE_ERANGE before anything is enqueued.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) with
 *     that device current, once; later calls on that device reuse it.
 *   - Every call shares the one array, which keeps the last call's tables; nothing in it has to
 *     start at zero, because each call rewrites everything its kernel reads.  Calls on the same
 *     stream are ordered; calls that overlap on the GPU (different streams, or several host
 *     threads on different streams) race on the array and must not be issued.  Host threads
 *     calling at once are serialised while the tables are written and copied.
 * Errors: TIDE_EINVAL (as tide_plan_layout and tide_reduce_scatter; no TIDE_FLAG_VEC_STRICT:
 * unaligned gradients take the element-wise path), TIDE_ERANGE as above or on int64 overflow,
 * TIDE_ECUDA, TIDE_ENOMEM (the host runtime failed to lock a mutex).  No C++ exception leaves it.
 */
int tide_reduce_scatter_noalloc(int32_t R, int32_t P, const int64_t *rows, const int64_t *row_len,
                                const void *const *grads, void *const *shards, void *stream);

/* ---- interference probes (measurement kernels of the interference harness) ----------------- */
/*
 * tide_probe_hold — launches `ctas` CTAs of `threads` threads, each claiming `smem_bytes` of
 * dynamic shared memory (so a large value keeps one CTA per SM, like a GEMM CTA), in clusters of
 * `cluster_size` (1..8), that keep their SM for `hold_ns` (<= 10 s).  Fig. 4's resident spin
 * kernels and Table 5's SM-id probe: with `records` (device, 3*ctas uint64) each CTA writes its
 * SM number and its %globaltimer values on arrival and departure, so CTAs that could not start in the first wave are
 * visible.  Asynchronous on `stream`; TIDE_EINVAL on bad sizes.
 */
int tide_probe_hold(int32_t ctas, int32_t threads, int32_t smem_bytes, int32_t cluster_size, uint64_t hold_ns,
                    uint64_t *records, void *stream);

/*
 * tide_probe_bulk_read — reads `bytes` of `buf` (16-byte aligned, device) with `ctas` CTAs, each
 * streaming `copy_bytes` bulk copies (multiple of 16) through `stages` shared-memory slots
 * (copy_bytes*stages <= 200 KB).  Measures how an SM's bulk-copy bandwidth depends on the copy
 * size.  out (device, 2 uint32): out[0] = XOR checksum of the first word of every copy, out[1] =
 * nonzero if a bounded wait (1 s) expired.
 */
int tide_probe_bulk_read(const void *buf, int64_t bytes, int32_t ctas, int32_t copy_bytes, int32_t stages,
                         uint32_t *out, void *stream);

/*
 * tide_probe_ingest — how many bytes per second one SM can bring in, the bound of any reduce-scatter
 * allowed only a few SMs (Fig. 4, Table 4: the pages' collectives hold 4 to 20 CTAs).  `ctas` CTAs
 * (each claims copy_bytes*stages of shared memory, so one per SM) read the device buffer `buf`
 * (256-byte aligned) in two parts at once:
 *   - [buf, buf + bulk_bytes): bulk copies of `copy_bytes` (multiple of 16) through `stages`
 *     shared-memory slots (copy_bytes*stages <= 231168 bytes, stages <= 16), each landed slot read out by
 *     `consumer_warps` warps, every 16-byte word (0: only its first word, the copy engine alone);
 *     whole copies only (bulk_bytes / copy_bytes of them);
 *   - the next ldg_bytes (a multiple of 32) from buf + round_up(bulk_bytes, 256): `ldg_warps` warps
 *     of 32-byte register loads, eight in flight per thread.
 * 1 + max(consumer_warps, 1) + ldg_warps <= 16.  The caller's buffer must hold both parts.
 * out (device, 2 uint32): out[0] ^= XOR checksum of what was read, out[1] |= 1 if a wait (1 s bound)
 * expired, 2 if copies were still landing 1 s after the last issue.  TIDE_EINVAL on bad arguments.
 */
int tide_probe_ingest(const void *buf, int64_t bulk_bytes, int64_t ldg_bytes, int32_t ctas, int32_t copy_bytes,
                      int32_t stages, int32_t consumer_warps, int32_t ldg_warps, uint32_t *out, void *stream);

/*
 * tide_probe_mixed — how reading and writing share one SM's traffic, the other half of the bound of
 * a reduce-scatter that may hold only a few SMs (it writes one fp32 sum per R bf16 values read).
 * `ctas` CTAs (one per SM: each claims copy_bytes*stages of shared memory) read [buf, buf +
 * bulk_bytes) as tide_probe_ingest's bulk part does (`consumer_warps` >= 1 warps read every 16-byte
 * word of each landed copy; buf 256-byte aligned) while `st_warps` warps per CTA write 32-byte
 * vectors into the CTA's equal share of [st_buf, st_buf + st_bytes) (st_buf 32-byte aligned,
 * st_bytes a multiple of 32), cycling over it until that CTA's reads have landed; with bulk_bytes
 * == 0 they write their share once.  With burst_rows > 0 the reading warps also write, as a
 * reduce-scatter stores its sums after the last rank's row: after every burst_rows landed copies
 * each reading thread stores burst_vecs 32-byte vectors (adjacent threads to adjacent vectors) into
 * the CTA's share, cycling over it.  The written values are a pattern of no meaning (the checked
 * pattern of the dedicated writers holds only when burst_rows == 0); nothing else is written.
 * 1 + consumer_warps + st_warps <= 16.
 * out (device, 3 uint64): out[0] ^= checksum of what was read, out[1] |= 1 if a wait (1 s bound)
 * expired, 2 if copies were still landing 1 s after the last issue, 4 if the writers stopped at
 * their 2 s bound; out[2] += bytes written.  TIDE_EINVAL on bad arguments.
 */
int tide_probe_mixed(const void *buf, int64_t bulk_bytes, void *st_buf, int64_t st_bytes, int32_t ctas,
                     int32_t copy_bytes, int32_t stages, int32_t consumer_warps, int32_t st_warps, int32_t burst_rows,
                     int32_t burst_vecs, uint64_t *out, void *stream);

/* ---- errors ------------------------------------------------------------------------------ */
const char *tide_strerror(int status);
/* cudaError_t code of the last CUDA failure reported as TIDE_ECUDA on this host thread. */
int tide_last_cuda_error(void);
/* Library version as major*10000 + minor*100 + patch. */
int tide_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TIDE_H */
