/*
 * moe.h - C ABI of the GB300 (sm_103a) MoE expert layer with tile-level return-copy overlap.
 *
 * The method is the one of the review page "Fine-grained Computation-Communication Overlap via
 * Tile-level Signaling and Scheduling for Mixture-of-Experts" (Cui, Wingkvist, Ericsson;
 * pith.science/paper/W2ZARMHG), cited here as [TLS] with the section of that page:
 *
 *   [TLS "The pith" / "Core claim"]      the return of expert outputs to the rank that sent each
 *        token need not wait for all expert compute: a persistent GEMM (producer) covering all
 *        experts publishes a readiness flag per output tile; a persistent copy kernel (consumer)
 *        on a small SM partition polls the flags and moves ready row bands to their owner.
 *   [TLS "What carries the argument"]    remote-owner-aligned row layout (rows grouped by expert,
 *        then by owner, each group padded to the tile height, so each tile has one owner),
 *        remote-first tile schedule (largest transfers first), row-band segments.
 *   [TLS "Load-bearing premise"] and [TLS "Referee Report", major comment 2, §3.3.1]  the tile
 *        must be visible before the flag is seen: here the producer's stores are released at GPU
 *        scope and the consumer acquires the flag before it reads.
 *   [TLS Figure 9 caption]               the sequential baseline: per-expert GEMM, then the bulk
 *        return copy, on identical inputs.
 *
 * On one GPU the R "ranks" are R logical owner partitions of the tokens: owner(t) = t / (T/R).
 * Each owner has a return buffer (a slice of Ret) in the same HBM; the "put" is a device copy.
 *
 * Conventions for every entry point
 *   - All arrays are row-major and contiguous. "device" pointers point to memory of the current
 *     CUDA device; "host" pointers to host memory (pinned for asynchronous copies).
 *   - bf16 arrays are passed as uint16_t bit patterns (IEEE bfloat16).
 *   - The caller owns every buffer and the stream. The library never allocates device memory,
 *     never frees anything and never synchronises the stream except in moe_status() (and
 *     moe_forward_dma, which waits on the host for the GPU's progress).
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default stream.
 *   - Return value: MOE_OK or a negative MOE_ERR_* code; no exception crosses the ABI, and the
 *     device never traps. moe_last_error() gives a message for the calling thread.
 *   - Work is enqueued on `stream`; results are valid once the stream has reached that point.
 *   - One workspace must not be used by two calls that can run at the same time.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_API __attribute__((visibility("default")))

/* ---- return codes ---------------------------------------------------------------------- */
#define MOE_OK 0
#define MOE_ERR_ARG (-1)       /* invalid config, NULL pointer, misaligned pointer          */
#define MOE_ERR_WORKSPACE (-2) /* workspace smaller than moe_workspace_size()               */
#define MOE_ERR_CUDA (-3)      /* a CUDA runtime / driver call failed (launch, copy, ...)   */
#define MOE_ERR_TIMEOUT (-4)   /* a bounded device wait ran out (reported by moe_status)    */
#define MOE_ERR_DEVICE (-5)    /* current device is not sm_103 / lacks the needed resources */
#define MOE_ERR_PLAN (-6)      /* a device-side bounds check on plan indices failed         */

/* ---- config flags ---------------------------------------------------------------------- */
#define MOE_PLAN_SKIP_PERMUTE 0x1u    /* moe_plan: stop after the plan, do not fill Xc        */
#define MOE_TAIL_ASSIST 0x2u          /* producer CTAs that finish their GEMM tiles join the  */
                                      /* copy (the consumer partition is unchanged)           */
#define MOE_COPY_WARPS 0x4u           /* copy engines also run as two extra warps in every    */
                                      /* producer CTA (16-byte loads/stores, no shared memory),*/
                                      /* so consumer_ctas may be 0: no SM leaves the GEMM       */
#define MOE_PAIR_UMMA 0x8u            /* expert GEMMs on CTA pairs: UMMA 256 x 256 over two SMs*/
                                      /* (tcgen05 cta_group::2), half the B tile per SM; the   */
                                      /* down-projection too when d % 256 == 0, consumer_ctas  */
                                      /* is even and MOE_COPY_WARPS is not set                 */
#define MOE_DIRECT_TAIL 0x10u         /* the down-projection's epilogue writes the bands that  */
                                      /* its work items with a tile among the launch's last    */
                                      /* tail_window tile positions (the last wave) complete   */
                                      /* straight into their owner's slice of Ret; the         */
                                      /* consumer skips them and their rows of Yp are not      */
                                      /* written                                               */
#define MOE_FUSED_DISPATCH 0x20u      /* the permute's row copies move into the SwiGLU GEMM:  */
                                      /* its epilogue warps copy the token rows into Xc,      */
                                      /* expert by expert, before their first tile and        */
                                      /* release a per-expert row count that the TMA threads  */
                                      /* acquire before loading an expert's rows; the permute */
                                      /* launch only computes the slots                       */
#define MOE_FUSED_GEMMS 0x40u         /* both expert GEMMs in one persistent launch on CTA     */
                                      /* pairs (needs the down-projection on pairs): SwiGLU   */
                                      /* tiles first; an expert's down-projection tiles start */
                                      /* once all its SwiGLU tiles have published; the        */
                                      /* consumer clusters take SwiGLU tiles, then copy       */
#define MOE_PDL 0x80u                 /* programmatic dependent launch between the layer's    */
                                      /* GEMMs and combine too (the routing, plan and permute */
                                      /* kernels always use it; the permute starts once the   */
                                      /* plan has published the row layout, beside the rest  */
                                      /* of it): each starts its prologue (barriers, TMEM,    */
                                      /* descriptor prefetch, plan tables) while the previous */
                                      /* one finishes and waits on the GPU before reading its */
                                      /* outputs (not for the cooperative single-CTA down-    */
                                      /* projection)                                          */
#define MOE_TEST_STALL_CONSUMER 0x100u /* test hook: consumers wait for a flag value that no  */
                                      /* producer writes, so their bounded wait runs out      */
#define MOE_TEST_PLAN_FAIL 0x200u     /* test hook: the plan kernel reports a failed bounds   */
                                      /* check (MOE_ERR_PLAN, detail -3) although the plan is */
                                      /* valid, to test that the status reaches the caller    */
#define MOE_TEST_STALL_LAYOUT 0x2000u /* test hook: the plan never publishes the row layout, */
                                      /* so the permute's bounded wait for it runs out        */
                                      /* (MOE_ERR_TIMEOUT) and it copies no row               */
#define MOE_ADAPTIVE_CONSUMERS 0x1000u /* the CTA-pair down-projection picks its consumer      */
                                      /* partition at run time from its tile count: the       */
                                      /* fewest producer pairs that finish the tiles in the    */
                                      /* fewest waves any partition with one or more consumer */
                                      /* pairs allows; every other pair copies (consumer_ctas */
                                      /* then only sizes the launch's default)                */
#define MOE_TEST_STALL_PIPE0 0x400u   /* test hooks: in the CTA-pair GEMMs the TMA thread of   */
#define MOE_TEST_STALL_PIPE1 0x800u   /* rank 0 (PIPE0) or rank 1 (PIPE1) of every pair stops  */
                                      /* issuing loads halfway through its first tile, so the */
                                      /* pair's bounded waits run out (MOE_ERR_TIMEOUT) and   */
                                      /* its abort path settles the loads still in flight     */

/*
 * Problem and knobs.
 *   T tokens, model width d, expert hidden width ffn, E experts, top-k = topk, R owners,
 *   tile_M = GEMM tile height tbM (each (expert, owner) group is padded to a multiple of it).
 *   consumer_ctas = c_CTA, the SMs given to the consumer ([TLS "Axiom & Free-Parameter Ledger"],
 *   swept 2-24 on the page); mgb = bands per interior segment (same section, 1 or 2 there).
 *   timeout_us bounds every device-side wait (0 = 2,000,000 us).
 *   tail_window (with MOE_DIRECT_TAIL): the number of the down-projection's last tile hand-out
 *   positions; the bands completed by work items with a tile among them are returned by the
 *   epilogue itself; 0 = one wave (one tile per producer CTA, or per producer CTA pair on CTA
 *   pairs).
 * Limits: d % 128 == 0, ffn % 128 == 0, 1 <= topk <= min(E, 8), 1 <= E <= 256, T % R == 0,
 *   E*R <= 1024, tile_M in {64, 128}, 1 <= mgb <= 4, 1 <= consumer_ctas <= SMs/2 (0 allowed
 *   with MOE_COPY_WARPS; checked at launch), tail_window >= 0, P_max < 2^30 (see moe_layout).
 */
typedef struct moe_config {
    int32_t T, d, ffn, E, topk, R, tile_M;
    int32_t consumer_ctas;
    int32_t mgb;
    uint32_t flags;
    uint32_t timeout_us;
    int32_t tail_window;
    int32_t reserved[4]; /* must be zero */
} moe_config;

/*
 * Byte offsets (from the workspace base) and sizes of the regions of a workspace. Every region
 * starts on a 1024-byte boundary. Shapes use P_max = the largest padded row count the routing can
 * produce, T*topk + min(E*R, T*topk)*(tile_M-1) rounded up to tile_M ([TLS "Referee Report",
 * major comment 1]: padding is per (expert, owner) group), and MT_max = P_max / tile_M.
 *
 * Two row layouts. The owner-aligned padded layout of the plan (rows `slot`, P rows, every
 * (expert, owner) group padded to tile_M) is the layout of the expert outputs Yp, so that each
 * output tile has one owner. The GEMM inputs Xc and Hc use the expert-compact layout (rows
 * `cslot`): the rows of each expert contiguous, its groups in owner order and each group's rows
 * in plan order, each expert's run padded with zero rows to a multiple of 128 (the UMMA tile
 * height); PC_max = T*topk + min(E, T*topk)*127 rounded up to 128. The SwiGLU GEMM then runs
 * whole 128-row tiles of one expert instead of padded owner groups.
 */
typedef struct moe_layout {
    size_t bytes;                     /* total workspace size                              */
    int32_t P_max, MT_max, n_chunks, chunk_tokens, n_tiles_n2, block_n2, rows_per_unit, units_per_band;
    int32_t PC_max, IU_max;           /* rows of Xc / Hc; SwiGLU work items (PC_max / 128)     */
    size_t idx;        /* int32 [T, topk]   expert of pair (t, j), descending logit            */
    size_t gate;       /* f32   [T, topk]   gate of pair (t, j)                                */
    size_t rank;       /* int32 [T, topk]   rank of t among the chunk's tokens routed to e     */
    size_t chunk_cnt;  /* int32 [n_chunks, E]                                                  */
    size_t chunk_base; /* int32 [n_chunks, E] rows of e in earlier chunks of the same owner    */
    size_t counts;     /* int32 [E, R]      n_{e,r} = |G_{e,r}|                                */
    size_t offsets;    /* int32 [E*R + 1]   first padded row of group e*R+r; last entry = P    */
    size_t ret_off;    /* int32 [R, E + 1]  exclusive prefix over e of n_{e,r}                 */
    size_t tiles;      /* int32 [MT_max, 4] (e, r, row0, valid) per M-tile, layout order       */
    size_t tile_ret;   /* int32 [MT_max]    row of Ret receiving the tile's first row          */
    size_t sched;      /* int32 [MT_max]    M-tile at each position of the remote-first        */
                       /*                   schedule: valid rows descending, ties in layout   */
                       /*                   order ([TLS "What carries the argument"])         */
    size_t order;      /* int32 [MT_max]    M-tile at each position of the down-projection's   */
                       /*                   hand-out order: the schedule re-sorted stably by  */
                       /*                   expert, most loaded (most rows) first, ties to    */
                       /*                   the lower id; the consumer copies in this order   */
    size_t seg;        /* int32 [MT_max, 2] (first position, bands) of each hand-out position's */
                       /*                   segment                                           */
    size_t experts;    /* int32 [E, 8]      first M-tile, M-tiles, first hand-out position,    */
                       /*                   hand-out rank, SwiGLU work items, first SwiGLU    */
                       /*                   item, first down-projection item, first Xc row    */
    size_t items_up;   /* int32 [IU_max, 2] SwiGLU work items: (first Xc row, expert), 128 rows */
    size_t items_down; /* int32 [MT_max, 2] down-projection work items: the SwiGLU items with   */
                       /*                   the experts in hand-out rank order                */
    size_t slot;       /* int32 [T, topk]   row of pair (t, j) in Yp (padded layout)            */
    size_t cslot;      /* int32 [T, topk]   row of pair (t, j) in Xc / Hc (compact layout)      */
    size_t ret_slot;   /* int32 [T, topk]   row of pair (t, j) in Ret                          */
    size_t yrow;       /* int32 [PC_max]    Yp row of each Xc / Hc row, -1 for a padding row    */
    size_t tile_crow;  /* int32 [MT_max]    Xc / Hc row of the first row of each M-tile (band) */
    size_t band_item;  /* int32 [MT_max]    down-projection work item holding each M-tile's last row */
    size_t tok_of;     /* int32 [PC_max]    token of each Xc / Hc row, -1 for a padding row     */
    size_t xrows;      /* uint32 [E]        rows of each expert copied into Xc (fused dispatch) */
    size_t xready;     /* uint32 [E]        SwiGLU tile quarters published per expert (fused)   */
    size_t meta;       /* int32 [64]        P, M-tiles, work counters, status (see csrc)       */
    size_t flags;      /* uint32 [MT_max, n_tiles_n2] rows of each tile stored (ready at its   */
                       /*                   valid rows)                                       */
    size_t bands;      /* uint32 [MT_max]   rows of each band stored over all its N tiles      */
                       /*                   (ready at valid rows x n_tiles_n2)                */
    size_t trace;      /* uint64 [16]       %globaltimer stamps of the last call (ns), [0, 8);  */
                       /*                   SM clock counters, [8, 12), zeroed by the caller  */
    size_t Xc;         /* bf16 [PC_max, d]  permuted tokens, expert-compact, zero padding rows */
    size_t Hc;         /* bf16 [PC_max, ffn] SwiGLU hidden, same rows                          */
    size_t Yp;         /* bf16 [P_max, d]   expert outputs                                     */
    size_t Ret;        /* bf16 [T*topk, d]  owner return buffers, R slices of (T/R)*topk rows  */
    size_t in_logits;  /* f32  [2, T, E]    staging for moe_forward_host(_pipelined), 2 slots   */
    size_t in_x;       /* bf16 [2, T, d]    staging for moe_forward_host(_pipelined), 2 slots   */
    size_t out;        /* f32  [2, T, d]    staging for moe_forward_host(_pipelined), 2 slots   */
} moe_layout;

/* Trace slots (uint64 ns, %globaltimer) written by the last moe_forward / _sequential call. */
#define MOE_TRACE_GEMM2_START 0  /* earliest start of a down-projection tile                 */
#define MOE_TRACE_GEMM2_END 1    /* latest readiness flag (overlapped) / tile end (sequential) */
#define MOE_TRACE_COPY_START 2   /* earliest start of a row-band copy                        */
#define MOE_TRACE_COPY_END 3     /* latest completion of a row-band copy                     */
#define MOE_TRACE_BAND_DONE 4    /* overlapped: latest time a band's last tile was published   */
#define MOE_TRACE_LAST_ACQUIRE 5 /* overlapped: latest time a copy engine acquired a band      */
#define MOE_TRACE_LAST_LOAD 6    /* latest issue of a bulk load by a copy engine               */
#define MOE_TRACE_LAST_DRAIN 7   /* latest start of a copy engine's final drain                */

/* Clock counters (uint64), summed over calls until the caller zeroes them (moe_plan leaves them):
 * CTA 0 of each expert-GEMM launch adds the cycles of its SM's clock (%clock64) and the %globaltimer
 * nanoseconds of one span, from the end of its wait for the previous kernel to the end of its tiles.
 * 1000 * cycles / ns is the mean SM clock in MHz over those launches. */
#define MOE_TRACE_UP_CYCLES 8    /* SwiGLU GEMM (both GEMMs in MOE_FUSED_GEMMS)                */
#define MOE_TRACE_UP_NS 9
#define MOE_TRACE_DOWN_CYCLES 10 /* down-projection                                          */
#define MOE_TRACE_DOWN_NS 11

/* Size in bytes of the workspace for `cfg` (host-only arithmetic, no CUDA call).
 * Returns MOE_ERR_ARG for an invalid config. */
MOE_API int moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Offsets of the workspace regions for `cfg` (host-only arithmetic). For tests and tools that
 * read the plan or the intermediates; the contents are valid after a call on the stream. */
MOE_API int moe_workspace_layout(const moe_config* cfg, moe_layout* out);

/*
 * moe_plan: router + layout, the first half of the forward pass.
 *   logits   device f32  [T, E]   router logits (finite)
 *   x        device bf16 [T, d]   tokens (may be NULL with MOE_PLAN_SKIP_PERMUTE)
 *   topk_idx device int32 [T, topk] or NULL: copy of the routing (experts, descending logit,
 *            ties to the lower expert id)
 *   topk_w   device f32 [T, topk] or NULL: gates, softmax over the k chosen logits
 *   ws       device workspace of ws_bytes >= moe_workspace_size(cfg), 256-byte aligned
 * Fills the workspace's idx, gate, counts, offsets, tiles, sched, seg, slot, cslot, ret_slot, ...
 * and (unless MOE_PLAN_SKIP_PERMUTE) Xc with zero padding rows. The histogram / scan / tile-owner map
 * follow [TLS "What carries the argument"]; the plan is built on the device, so no host round
 * trip is needed before the GEMMs ([TLS "Referee Report", minor comment 4, §2.2]).
 */
MOE_API int moe_plan(const moe_config* cfg, const float* logits, const uint16_t* x, int32_t* topk_idx,
                     float* topk_w, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward: the whole MoE layer with the tile-level overlapped return copy.
 *   logits device f32 [T, E]; x device bf16 [T, d];
 *   W1, W3 device bf16 [E, ffn, d] (gate and up projections, K-major);
 *   W2     device bf16 [E, d, ffn] (down projection, K-major);
 *   out    device f32 [T, d]: out[t] = sum_j gate[t, j] * FFN_{idx[t, j]}(x[t]),
 *          FFN_e(v) = W2_e (silu(W1_e v) * (W3_e v));
 *   ws     workspace as in moe_plan. Weights and x are only read; 16-byte aligned pointers.
 * Steps on `stream`: route, plan, permute, SwiGLU grouped GEMM over all experts (one persistent
 * launch), then one persistent launch in which all but consumer_ctas CTAs run the down-projection
 * GEMM, tiles handed out in the hand-out order (the remote-first schedule re-sorted by expert: see
 * moe_layout.order; on CTA pairs, where one expert's W2 is at least 64 MB and its rows of the hidden
 * activations at most 64 MB, the expert's tiles go N tile by N tile over its bands, the last
 * expert's band by band), and release a flag per finished tile while the last consumer_ctas CTAs
 * acquire the flags and copy each ready segment of row bands into its owner's slice of Ret, then
 * the weighted top-k combine. Flags: MOE_TAIL_ASSIST (producers that finished join the copy),
 * MOE_COPY_WARPS (copy engines also inside every producer CTA; consumer_ctas may be 0),
 * MOE_PAIR_UMMA (the expert GEMMs on CTA pairs), MOE_DIRECT_TAIL (the last wave's bands written into
 * Ret by the epilogue); none changes out or Ret, bit for bit. A bounded wait that runs out, or a plan
 * entry that fails its bounds check, is reported by moe_status(), not here.
 */
MOE_API int moe_forward(const moe_config* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                        const uint16_t* W3, const uint16_t* W2, float* out, void* ws, size_t ws_bytes,
                        void* stream);

/*
 * moe_forward_sequential: same arguments and result as moe_forward; the down-projection GEMM runs
 * on all SMs without flags, then the return copy runs on all SMs, then the combine. This is the
 * GEMM-then-copy baseline of [TLS Figure 9 caption]; the two GEMM launches use the same tile code,
 * so its out, Yp and Ret are bitwise equal to moe_forward's.
 */
MOE_API int moe_forward_sequential(const moe_config* cfg, const float* logits, const uint16_t* x,
                                   const uint16_t* W1, const uint16_t* W3, const uint16_t* W2, float* out,
                                   void* ws, size_t ws_bytes, void* stream);

/*
 * moe_copy_only: the return copy alone (every valid row of every band of Yp into its owner's slice
 * of Ret, 16 KB TMA bulk copies through shared memory) on `ctas` CTAs, one per SM, for measuring
 * the copy's bandwidth against the size of the consumer partition ([TLS "What carries the
 * argument"]: the consumer's SM budget c_CTA). Uses the plan and Yp of the last moe_forward /
 * moe_forward_sequential on `ws`; writes only Ret and a work counter. 1 <= ctas <= SMs, else
 * MOE_ERR_ARG.
 */
MOE_API int moe_copy_only(const moe_config* cfg, void* ws, size_t ws_bytes, int ctas, void* stream);

/*
 * moe_forward_ex: moe_forward (sequential == 0) or moe_forward_sequential (sequential != 0) that
 * also records caller-created CUDA events (cudaEvent_t passed as void*) on `stream` between the
 * launches, for per-stage timing; stage_events may be NULL, and so may any entry:
 *   [MOE_EV_BEGIN]     before routing            [MOE_EV_PLANNED] after the permute
 *   [MOE_EV_UP]        after the SwiGLU GEMM     [MOE_EV_DOWN]    after the down-projection launch
 *                                                                 (overlapped: GEMM + return copy)
 *   [MOE_EV_COPIED]    after the return copy (overlapped: same point as MOE_EV_DOWN)
 *   [MOE_EV_END]       after the combine
 * With MOE_FUSED_GEMMS (one launch for both GEMMs) MOE_EV_UP, MOE_EV_DOWN and MOE_EV_COPIED all
 * follow that launch.
 * While `stream` is being captured into a CUDA graph, each record becomes an event-record node of
 * the graph (cudaEventRecordExternal), recorded again by every replay.
 */
#define MOE_EV_BEGIN 0
#define MOE_EV_PLANNED 1
#define MOE_EV_UP 2
#define MOE_EV_DOWN 3
#define MOE_EV_COPIED 4
#define MOE_EV_END 5
#define MOE_EV_COUNT 6
MOE_API int moe_forward_ex(const moe_config* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                           const uint16_t* W3, const uint16_t* W2, float* out, void* ws, size_t ws_bytes,
                           int sequential, void* const* stage_events, void* stream);

/*
 * moe_forward_host: moe_forward with host inputs and output, the call a serving process makes per
 * batch with weights resident on the device. logits_h (f32 [T, E]) and x_h (bf16 [T, d]) are copied
 * into the workspace's staging regions, the layer runs, and out_h (f32 [T, d]) receives the result;
 * all on `stream` (use pinned host memory for asynchronous copies). out_h is valid once the stream
 * has reached the end of this call. `sequential` != 0 selects the GEMM-then-copy baseline.
 */
MOE_API int moe_forward_host(const moe_config* cfg, const float* logits_h, const uint16_t* x_h,
                             const uint16_t* W1, const uint16_t* W3, const uint16_t* W2, float* out_h,
                             void* ws, size_t ws_bytes, int sequential, void* stream);

/*
 * moe_forward_host_pipelined: `steps` independent batches of the same shape through the layer,
 * each with its own host inputs and output (arrays of `steps` host pointers; pinned memory), with
 * the transfers of neighbouring batches overlapped with the layer: the inputs of batch i+1 are
 * copied in and the output of batch i-1 is copied out on two internal streams while batch i runs
 * on `stream`, through two staging slots in the workspace. With steps > 1 the layer's launches for
 * each slot are captured once as a CUDA graph (kept for the last 4 (config, workspace, weights)
 * combinations per device) and replayed. Results equal `steps` calls of moe_forward_host. Not for
 * concurrent use from several host threads (the copy streams, events and graphs are per device). Every out_h[i] is valid once `stream` has reached the end of this call; the
 * host inputs must stay unchanged until then. No counterpart in the method's pages: the serving
 * loop around the layer.
 */
MOE_API int moe_forward_host_pipelined(const moe_config* cfg, int steps, const float* const* logits_h,
                                       const uint16_t* const* x_h, const uint16_t* W1, const uint16_t* W3,
                                       const uint16_t* W2, float* const* out_h, void* ws, size_t ws_bytes,
                                       int sequential, void* stream);

/*
 * moe_forward_dma: moe_forward with the return copy on the GPU's copy engines (DMA) instead of SMs,
 * the DMA-offload idea of the FiCCO page ("Design Space Exploration of DMA based Finer-Grain Compute
 * Communication Overlap", "Core claim": offloading communication to the GPU's DMA engines reduces
 * its contention with compute). Same arguments, result (out, Ret, bit for bit) and workspace as
 * moe_forward, plus:
 *   host_rec     pinned host memory mapped into the device (e.g. cudaHostAlloc, or any page-locked
 *                memory on a system with unified addressing), 16-byte aligned, host_bytes >=
 *                moe_dma_host_bytes(cfg). Owned by the caller; not to be used by two calls at once.
 *   stage_events as in moe_forward_ex (may be NULL); [MOE_EV_COPIED] is recorded on the library's
 *                copy stream after the last band's copy.
 * The down-projection runs on every SM (consumer_ctas, MOE_TAIL_ASSIST, MOE_COPY_WARPS and
 * MOE_ADAPTIVE_CONSUMERS are ignored); the epilogue warp that completes a band writes a record (its Yp row, Ret row and valid
 * rows, tagged with the call) into host_rec with a system-scope release. With MOE_DIRECT_TAIL the
 * bands the last wave completes are written into Ret by the epilogue and their records carry 0 rows
 * (nothing to copy). The calling
 * thread polls the records and issues one cudaMemcpyAsync per ready band (one per run of ready bands
 * that are adjacent in both Yp and Ret), device to device, on a copy stream of the library's own,
 * which starts after the work enqueued on `stream` before this call; `stream` waits for that copy
 * stream before the combine. So this call returns only after the
 * down-projection has finished on the GPU (it blocks for the layer's GEMMs) and cannot be captured
 * into a CUDA graph (MOE_ERR_ARG while `stream` is capturing). If the down-projection stops early (a
 * bounded wait ran out), the call sees the stream finish with records missing and returns
 * MOE_ERR_TIMEOUT; moe_status then gives the device status.
 */
MOE_API int moe_dma_host_bytes(const moe_config* cfg, size_t* bytes);
MOE_API int moe_forward_dma(const moe_config* cfg, const float* logits, const uint16_t* x, const uint16_t* W1,
                            const uint16_t* W3, const uint16_t* W2, float* out, void* ws, size_t ws_bytes,
                            void* host_rec, size_t host_bytes, void* const* stage_events, void* stream);

/*
 * moe_status: synchronises `stream`, then reads the device status word of the last call that used
 * `ws`. Returns MOE_OK, MOE_ERR_TIMEOUT (a flag or pipeline wait ran out; *detail = where) or
 * MOE_ERR_PLAN (a bounds check on plan indices failed). The word is cleared by the next call.
 * detail may be NULL. With ws == NULL it reads the status of the last moe_route_static call on the
 * current device instead (cfg must be that call's config; it allocates nothing either).
 */
MOE_API int moe_status(const moe_config* cfg, const void* ws, void* stream, int32_t* detail);

/* Number of SMs of the current device and whether it is supported (sm_103); host query only. */
MOE_API int moe_device_info(int32_t* sm_count, int32_t* supported);

/*
 * moe_route_static: routing and the row layout for callers that cannot allocate device memory and so
 * cannot provide moe_plan's workspace: code running inside a custom allocator's callback, a plugin
 * whose host application owns all device memory and hands none out, or a serving runtime whose
 * memory pool is fixed at start-up and may not grow while requests are in flight.
 * The paper has no counterpart of this entry point; it is a deployment convenience.
 *   logits   device f32 [T, E]  (input, as in moe_plan)
 *   topk_idx device int32 [T, topk], topk_w device f32 [T, topk]: the routing (as moe_plan's)
 *   slot, ret_slot device int32 [T, topk]: row of pair (t, j) in the padded layout / the return
 *            buffer; offsets device int32 [E*R + 1]: first padded row of each (expert, owner) group
 *            and the padded total P (all as in the workspace written by moe_plan)
 * It allocates nothing: its internal scratch (ranks, per-chunk counts, tile map, schedule, status)
 * is a file-scope device array of MOE_STATIC_SCRATCH_BYTES that every GPU which loads the library
 * holds until the process exits. A config whose scratch would exceed that size returns MOE_ERR_ARG
 * with the needed size in moe_last_error(). The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, once per CUDA context); make that first call before any stream
 * capture. All calls share the one array and each call overwrites what it reads: calls that can
 * overlap on the GPU (two streams, or two host threads) race and must be serialised by the caller.
 * cfg->flags has no effect here (no token rows are moved, so MOE_PLAN_SKIP_PERMUTE changes nothing),
 * except the test hook MOE_TEST_PLAN_FAIL. A plan entry that fails its device-side bounds check is
 * reported by moe_status(cfg, NULL, stream, &detail), which reads this call's status words from the
 * same array.
 */
#define MOE_STATIC_SCRATCH_BYTES (4 << 20)
MOE_API int moe_route_static(const moe_config* cfg, const float* logits, int32_t* topk_idx, float* topk_w,
                             int32_t* slot, int32_t* ret_slot, int32_t* offsets, void* stream);

/* Message of the last error on the calling thread ("" if none). The pointer stays valid until
 * the thread's next call into the library. */
MOE_API const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
