// Internal definitions shared by the kernels and the host side of libmoe.
// Hand-written inline PTX for sm_103a: mbarrier, TMA (cp.async.bulk.tensor), bulk copies,
// tcgen05 (TMEM allocation, UMMA, TMEM loads) and GPU-scope release/acquire.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

#include "../../include/moe.h"

namespace moe {

// ---- meta word indices (int32 [64] in the workspace) -------------------------------------
enum Meta : int {
    META_P = 0,            // padded rows P of this call
    META_MTILES = 1,       // M-tiles = P / tile_M
    META_UNITS = 2,        // copy units = M-tiles * units_per_band
    META_QUEUE = 3,        // next copy unit to hand out (overlapped consumer)
    META_QUEUE_SEQ = 4,    // next copy unit to hand out (sequential copy)
    META_STATUS = 5,       // 0 or a Status code (first error wins)
    META_STATUS_DETAIL = 6,
    META_ITEMS = 7,        // down-projection work items (128 compact rows of one expert)
    META_ITEMS_UP = 8,     // SwiGLU work items (128 rows of one expert in the compact layout)
    META_PC = 9,           // rows of the compact layout used by this call
    META_PRODUCERS = 10,   // producer CTAs of the last overlapped CTA-pair down-projection
    META_LAYOUT = 16,      // 1 once the plan has published the row layout the permute reads
    META_DISPATCH = 24,    // next block of compact rows to copy (MOE_FUSED_DISPATCH)
    META_TILES_UP = 32,    // next SwiGLU GEMM tile to hand out (single-CTA kernel), minus the grid
    META_TILES_DOWN = 48,  // next down-projection tile to hand out, minus the producer count
                           // (both on a 128-byte line away from the copy queues' line)
    META_COUNT = 64,
};

enum Status : int {
    ST_OK = 0,
    ST_FLAG_TIMEOUT = 1,   // consumer gave up waiting on a tile flag
    ST_PIPE_TIMEOUT = 2,   // an mbarrier wait of the GEMM pipeline gave up
    ST_COPY_TIMEOUT = 3,   // a bulk copy did not complete in time
    ST_BAD_PLAN = 4,       // a plan index failed its bounds check
    ST_PAIR_TMEM = 5,      // the two CTAs of a pair got different TMEM column bases
    ST_LAYOUT_TIMEOUT = 6, // the permute gave up waiting for the plan's row layout
};

// Trace slots (uint64): [0, TR_STEP) are the public per-call stamps, reset by the plan kernel;
// [TR_STEP, TR_COUNT) the clock counters, which the caller zeroes.
enum Trace : int { TR_STEP = 8, TR_COUNT = 16 };

// ---- GEMM geometry --------------------------------------------------------------------------
constexpr int BM = 128;            // UMMA M (rows of one MMA tile)
constexpr int BK = 64;             // K per pipeline stage: 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_STAGE_BYTES = 256 * BK * 2;            // 32 KB (up to N = 256)
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int GEMM_THREADS = 192;                      // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int GEMM_WARPS = GEMM_THREADS / 32;
constexpr int COPY_WARPS_EXTRA = 2;                    // copy-engine warps added with MOE_COPY_WARPS
constexpr int GEMM_THREADS_MAX = GEMM_THREADS + 32 * COPY_WARPS_EXTRA;
constexpr int TILE_Q = 4;          // slots of the tile hand-out ring (TMA thread -> UMMA issuer, epilogue)
constexpr int PAIR_TILE_Q = 8;     // the CTA-pair kernel's ring (>= PAIR_STAGES + 2, see gemm.cu)
constexpr int MISC_BYTES = 6144;  // barriers, flags and the expert table (4E+1 ints)
// epilogue staging: per epilogue warp two 32-row x 32-column bf16 chunks (2 KB each), written to
// global memory by TMA tensor stores
constexpr int EPI_CHUNK = 32;
constexpr int EPI_CHUNK_BYTES = 32 * EPI_CHUNK * 2;
constexpr int EPI_BYTES = 4 * 2 * EPI_CHUNK_BYTES;
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + EPI_BYTES + MISC_BYTES + 1024;  // + alignment slack
constexpr int TMEM_COLS = 512;                         // two 256-column fp32 accumulators
// CTA-pair GEMM (tcgen05 cta_group::2, UMMA 256 x 256 x 16 over two SMs): each CTA stages its own
// 128 token rows of A and one half (128 rows) of the 256-row B tile, so per k-block an SM writes
// and reads 32 KB of shared memory instead of 48 KB.
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_A_BYTES = BM * BK * 2;              // 16 KB
constexpr int PAIR_B_BYTES = 128 * BK * 2;             // 16 KB
constexpr int PAIR_STAGE_BYTES = PAIR_A_BYTES + PAIR_B_BYTES;
constexpr int PAIR_SMEM = PAIR_STAGES * PAIR_STAGE_BYTES + EPI_BYTES + MISC_BYTES + 1024;
static_assert(PAIR_SMEM <= 227 * 1024, "pair GEMM shared memory");
// the fused launch of both GEMMs (MOE_FUSED_GEMMS) keeps two expert tables and the SwiGLU tile counts
constexpr int PAIR_SMEM_FUSED = PAIR_SMEM + 4096;
static_assert(PAIR_SMEM_FUSED <= 227 * 1024, "fused pair GEMM shared memory");
constexpr int BN1 = 128;                               // output columns of a SwiGLU tile
constexpr int MAX_E = 256;

// copy engines of the consumer (one per warp, two staging buffers each, in the stage area)
constexpr int COPY_PIECE = 16384;
constexpr int COPY_WARPS = GEMM_THREADS / 32;                    // 6
constexpr int COPY_NBUF = 2 * COPY_WARPS;                        // 12 buffers / mbarriers
static_assert(COPY_NBUF * COPY_PIECE <= STAGES * STAGE_BYTES, "copy staging must fit the stage area");
constexpr int UNIT_BYTES = 65536;                      // target bytes of one copy unit
constexpr int TAIL_UNIT_BYTES = COPY_PIECE;            // units of the last bands: one piece each
constexpr int TAIL_TILES = 320;                        // tiles of the last bands (about two waves)

// ---- parameters passed by value to kernels --------------------------------------------------
struct PlanPtrs {
    int32_t* idx;
    float* gate;
    int32_t* rank;
    int32_t* chunk_cnt;
    int32_t* chunk_base;
    int32_t* counts;
    int32_t* offsets;
    int32_t* ret_off;
    int32_t* tiles;      // [MT_max][4]
    int32_t* tile_ret;
    int32_t* sched;      // remote-first schedule (bands by valid rows, descending)
    int32_t* order;      // hand-out order of the down-projection and the copy (band at each position)
    int32_t* seg;        // [MT_max][2] segment of each hand-out position
    int32_t* experts;    // [E][8]: first M-tile, M-tiles, first hand-out position, hand-out rank,
                         //         SwiGLU items, first SwiGLU item, first down item, first Xc row
    int32_t* items_up;   // [IU_max][2] SwiGLU work items (first Xc row, expert), experts in id order
    int32_t* items_down; // [MT_max][2] the SwiGLU items, experts in hand-out rank order
    int32_t* slot;       // padded-layout row (Yp) of each (token, choice)
    int32_t* cslot;      // compact-layout row (Xc, Hc) of each (token, choice)
    int32_t* ret_slot;
    int32_t* yrow;       // [PC_max] Yp row of each compact row, -1 for a padding row
    int32_t* tile_crow;  // [MT_max] compact row of each band's first row
    int32_t* band_item;  // [MT_max] down-projection work item holding each band's last row
    int32_t* meta;
    uint32_t* flags;
    uint32_t* bands;
    unsigned long long* trace;
    uint32_t* host_rec;  // moe_forward_dma: band records in mapped pinned host memory (else null)
    const __nv_bfloat16* x;  // tokens [T, d] (MOE_FUSED_DISPATCH: read by the SwiGLU GEMM)
    int32_t* tok_of;     // [PC_max] token of each compact row, -1 for a padding row
    uint32_t* xrows;     // [E] compact rows of each expert copied so far (MOE_FUSED_DISPATCH)
    uint32_t* xready;    // [E] SwiGLU tile quarters of each expert published (MOE_FUSED_GEMMS)
    __nv_bfloat16* Xc;
    __nv_bfloat16* Hc;
    __nv_bfloat16* Yp;
    __nv_bfloat16* Ret;
};

struct Shape {
    int T, d, ffn, E, k, R, tbM;
    int mgb;
    int chunk_tokens, n_chunks;
    int P_max, MT_max;
    int PC_max, IU_max;             // compact rows and SwiGLU work items (PC_max / 128)
    int bn2, n_tiles_n2;            // down-projection N tile and N tiles per band
    int rows_per_unit, units_per_band;           // copy units of the leading bands
    int rows_per_unit_tail, units_per_band_tail;  // ... and of the last tail_bands bands
    int tail_bands;
    int down_n_outer_items;         // pair down-projection: experts of at most this many items
                                    // take their tiles N tile by N tile (0: none)
    int tail_window;                // MOE_DIRECT_TAIL: hand-out positions of the direct window (0: one wave)
    uint32_t host_epoch;            // moe_forward_dma: the call's tag of its host records
    unsigned long long timeout_ns;
    uint32_t flags;
};

// ---- host-side launchers (defined in the .cu files) ------------------------------------------
cudaError_t launch_route(const Shape& s, const float* logits, const PlanPtrs& p, cudaStream_t st);
cudaError_t launch_plan(const Shape& s, const PlanPtrs& p, cudaStream_t st);
cudaError_t launch_permute(const Shape& s, const __nv_bfloat16* x, const PlanPtrs& p, int sms, cudaStream_t st);
// tmA: 128-row boxes of the compact token rows
cudaError_t launch_gemm_swiglu(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmW1,
                               const CUtensorMap& tmW3, const CUtensorMap& tmOut, int sms, cudaStream_t st);
// The same SwiGLU GEMM on CTA pairs (cluster of 2, UMMA M = 256); grid = 2 x co-resident pairs.
cudaError_t launch_gemm_swiglu_pair(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA,
                                    const CUtensorMap& tmW1, const CUtensorMap& tmW3, const CUtensorMap& tmOut,
                                    cudaStream_t st);
// tmA: 128-row boxes of the compact hidden rows; tmOut: 32 x 32 boxes of Yp
cudaError_t launch_gemm_down(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmW2,
                             const CUtensorMap& tmOut, int sms, int consumers, bool overlapped, cudaStream_t st);
// The down-projection on CTA pairs (tmW2h: 128-row boxes of W2; needs bn2 = 256, consumers even, no
// copy warps); grid = 2 x co-resident pairs.
cudaError_t launch_gemm_down_pair(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmW2h,
                                  const CUtensorMap& tmOut, int consumers, bool overlapped, cudaStream_t st);
// Both expert GEMMs in one launch on CTA pairs (MOE_FUSED_GEMMS): SwiGLU operands (Xc, W1, W3, Hc
// store) and down-projection operands (Hc, W2 halves, Yp store); the last `consumers` (even) CTAs
// copy once the SwiGLU tiles are gone.
cudaError_t launch_gemm_fused_pair(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmXc, const CUtensorMap& tmW1,
                                   const CUtensorMap& tmW3, const CUtensorMap& tmHcOut, const CUtensorMap& tmHc,
                                   const CUtensorMap& tmW2h, const CUtensorMap& tmYpOut, int consumers,
                                   cudaStream_t st);
cudaError_t launch_copy_seq(const Shape& s, const PlanPtrs& p, int sms, cudaStream_t st);
cudaError_t launch_combine(const Shape& s, const PlanPtrs& p, float* out, int sms, cudaStream_t st);

// Launch with or without programmatic dependent launch (PDL, MOE_PDL): with it the kernel may start
// before the previous kernel on the stream has finished; it must call griddep_wait() before it
// touches that kernel's outputs (every kernel launched this way does, after its prologue).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                           Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Copy units of a call with MT bands: the last min(tail_bands, MT) bands in hand-out order are cut
// into smaller units than the others, so the copy after the last tile spreads over more engines.
__host__ __device__ inline int copy_unit_count(const Shape& s, int MT) {
    const int tb = MT < s.tail_bands ? MT : s.tail_bands;
    return (MT - tb) * s.units_per_band + tb * s.units_per_band_tail;
}
// Unit u -> (hand-out position, first row within the band, rows per unit of that band).
__host__ __device__ inline void copy_unit_decode(const Shape& s, int MT, int u, int* pos, int* rb, int* rpu) {
    const int tb = MT < s.tail_bands ? MT : s.tail_bands;
    const int lead = (MT - tb) * s.units_per_band;
    if (u < lead) {
        *pos = u / s.units_per_band;
        *rb = (u - *pos * s.units_per_band) * s.rows_per_unit;
        *rpu = s.rows_per_unit;
    } else {
        const int v = u - lead, q = v / s.units_per_band_tail;
        *pos = (MT - tb) + q;
        *rb = (v - q * s.units_per_band_tail) * s.rows_per_unit_tail;
        *rpu = s.rows_per_unit_tail;
    }
}

// ============================================================================================
// Device primitives
// ============================================================================================
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// SM clock of a launch: one thread notes its SM's cycle counter and the global timer at the start
// of the span and adds both differences to a pair of trace counters at its end; summed cycles over
// summed nanoseconds is the mean SM clock over the launches (all SMs share one clock).
struct ClockSpan {
    long long cycles;
    unsigned long long ns;
    bool on;
};
__device__ __forceinline__ ClockSpan clock_span_start(bool on) {
    ClockSpan c{0, 0, on};
    if (on) {
        c.cycles = clock64();
        c.ns = globaltimer();
    }
    return c;
}
__device__ __forceinline__ void clock_span_add(const PlanPtrs& p, const ClockSpan& c, int slot) {
    if (!c.on) return;
    atomicAdd(&p.trace[slot], (unsigned long long)(clock64() - c.cycles));
    atomicAdd(&p.trace[slot + 1], globaltimer() - c.ns);
}

// Programmatic dependent launch: wait until the grids this launch depends on have completed and
// their writes are visible (a no-op for a launch without a programmatic dependency), and let the
// next launch on the stream start its prologue (it waits the same way before reading ours).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Record the first error of a call in the status word.
__device__ __forceinline__ void set_status(int32_t* meta, int code, int detail) {
    if (atomicCAS(&meta[META_STATUS], 0, code) == 0) atomicExch(&meta[META_STATUS_DETAIL], detail);
}

// ---- mbarrier ------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// Complete `bytes` transaction bytes on `bar` without a copy: settles a phase that expects bytes of
// loads that were never issued.
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `bar` with the given parity to complete. Gives up (returns
// false) after timeout_ns of %globaltimer or when another role has raised *abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long timeout_ns,
                                          volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > timeout_ns) return false;
        }
    }
}

// ---- TMA -----------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// shared -> global tensor store of one box, tracked as a bulk async-group of the issuing thread
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, const void* src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// ---- untiled bulk copies (global <-> shared) --------------------------------------------------
__device__ __forceinline__ void bulk_load(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(src_gmem)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst_gmem, const void* src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                     reinterpret_cast<uint64_t>(dst_gmem)),
                 "r"(smem_u32(src_smem)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make generic-proxy global writes observed by this thread visible to its later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- GPU-scope release / acquire -----------------------------------------------------------------
// System-scope release store (host-visible word of mapped pinned memory).
__device__ __forceinline__ void st_release_sys(uint32_t* p, uint32_t v) {
    asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// moe_forward_dma: tell the host that band m is complete: its Yp row, Ret row and valid rows (0 for a
// band the epilogue wrote into Ret itself, MOE_DIRECT_TAIL: nothing to copy), then the call's tag,
// released at system scope after a system-scope fence (the band's rows were made visible at GPU
// scope by every warp that stored them, and this warp's counter update came last).
__device__ __forceinline__ void host_band_record(const Shape& s, const PlanPtrs& p, int m, bool direct) {
    uint32_t* rec = p.host_rec + 4 + 4 * (size_t)m;
    __threadfence_system();
    rec[1] = (uint32_t)p.tile_ret[m];
    rec[2] = direct ? 0u : (uint32_t)p.tiles[4 * m + 3];
    rec[3] = (uint32_t)p.tiles[4 * m + 2];
    __threadfence_system();
    st_release_sys(rec, s.host_epoch);
}
__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_acq_rel_gpu_add(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Bounded wait until the GPU-scope word *w is non-zero (acquire); false after timeout_ns.
__device__ __forceinline__ bool wait_word(const uint32_t* w, unsigned long long timeout_ns) {
    if (ld_acquire_gpu(w)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        __nanosleep(64);
        if (ld_acquire_gpu(w)) return true;
        if (globaltimer() - t0 > timeout_ns) return false;
    }
}

// ---- tcgen05 ---------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulate, one thread issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Instruction descriptor of kind::f16: D f32, A and B bf16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
    return (1u << 4)                              // D format: f32
           | (1u << 7)                            // A format: bf16
           | (1u << 10)                           // B format: bf16
           | (uint32_t(N >> 3) << 17)             // N / 8
           | (uint32_t(M >> 4) << 24);            // M / 16
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 bytes, groups of
// 8 rows 1024 bytes apart (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B and a 64-element
// bf16 inner box). Tile bases are 1024-byte aligned, so the base-offset field is 0.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= uint64_t((smem_addr & 0x3FFFF) >> 4);    // start address / 16
    d |= uint64_t(1) << 16;                       // leading byte offset (unused by swizzled K-major)
    d |= uint64_t(1024 >> 4) << 32;               // stride byte offset: 8 rows * 128 B
    d |= uint64_t(1) << 46;                       // descriptor version of tcgen05
    d |= uint64_t(2) << 61;                       // layout: SWIZZLE_128B
    return d;
}

// 32 lanes x 32 columns of 32-bit TMEM data into 32 registers per thread, then wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// ---- CTA pairs (clusters of two) -------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Address in CTA `rank`'s shared memory of the variable at shared::cta address `addr` of this CTA.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Every thread of both CTAs: release this thread's prior memory operations, wait for all. Also
// the first step before any access to the peer's shared memory (the peer has started).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Store a 32-bit value into a peer CTA's shared memory; the store completes as 4 transaction bytes
// on the peer's mbarrier (both addresses in the peer CTA, from mapa).
__device__ __forceinline__ void st_async_u32(uint32_t cluster_addr, uint32_t v, uint32_t cluster_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.u32 [%0], %1, [%2];" ::"r"(cluster_addr),
                 "r"(v), "r"(cluster_bar)
                 : "memory");
}
// Arrive on a barrier of the pair (own or peer) with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// mbar_wait for a barrier that the peer CTA arrives on (cluster-scope acquire).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, unsigned long long timeout_ns,
                                                  volatile int* abort) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > timeout_ns) return false;
        }
    }
}
// tcgen05 with cta_group::2: one warp of each CTA of the pair allocates / frees together (both
// get the same column base); one thread of the even CTA issues the UMMAs, which read A rows and
// B halves from the same shared-memory offsets in both CTAs and write each CTA's own TMEM lanes.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at `bar`'s offset in every CTA of `mask` when the UMMAs issued so far
// by this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// TMA tile load into this CTA's shared memory whose completion (complete_tx) is signalled on an
// mbarrier of either CTA of the pair (cta_group::2): the odd CTA's operand loads complete on the
// even CTA's stage barrier, which the UMMA issuer waits on.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x,
                                                 int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x, int y,
                                                 int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
        "%3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

#endif  // __CUDACC__

}  // namespace moe
