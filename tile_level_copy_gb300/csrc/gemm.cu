// Persistent grouped expert GEMMs on tcgen05 (fp32 accumulators in TMEM), fed by TMA through a
// shared-memory ring, with warp-specialised roles:
//   warp 0      one thread issues the TMA loads of A (token rows) and B (expert weights)
//   warp 1      allocates 512 TMEM columns; one thread issues the UMMAs (two accumulators, so the
//               epilogue of tile i overlaps the main loop of tile i+1)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, conversion, staging in shared memory and
//               TMA tensor stores of 32 x 32 chunks to global memory
//   warps 6-7   (down-projection with MOE_COPY_WARPS) SIMT copy engines of the return copy
// gemm_kernel<1|2> is the single-CTA kernel (UMMA 128 x N x 16, 4-stage ring); gemm_pair_kernel<1|2>
// runs either GEMM on CTA pairs (UMMA 256 x 256 x 16, cta_group::2, 6-stage ring per CTA). Tiles are
// handed out at run time from a counter per GEMM (see "Tile hand-out" below).
//
// Method: "Fine-grained Computation-Communication Overlap via Tile-level Signaling and Scheduling
// for Mixture-of-Experts" (pith.science/paper/W2ZARMHG):
//   "Core claim" - one rank-wide persistent GEMM covers all experts in one launch and publishes a
//       readiness flag after each tile's epilogue store;
//   "Load-bearing premise" and "Referee Report" major comment 2 (§3.3.1) - the tile must be
//       visible before the flag: each of the four epilogue warps waits until its stores of the
//       tile have completed, fences the async proxy, then adds its rows to the tile flag and to
//       the band's counter with release semantics; copy engines read the band counter with
//       ld.acquire.gpu (ready at valid rows x tiles per band); bulk engines fence the async proxy
//       first.
//   "What carries the argument" - the consumer runs on a small dedicated SM partition; here the
//       partition is the last consumer_ctas CTAs of the down-projection's own launch (a cooperative
//       launch for the single-CTA kernel, so producers and consumers are co-resident; the pair
//       kernel hands out every tile at run time, so no band waits for a particular CTA).
#include "copy_ring.cuh"

namespace moe {

struct Smem {
    uint8_t* stages;
    uint8_t* epi;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint64_t* cbar;
    uint64_t* tq_full;   // tile hand-out ring: slot written (count 1)
    uint64_t* tq_empty;  // slot read by the UMMA issuer and the 4 epilogue warps (count 5)
    uint32_t* tmem_base;
    volatile int* abort;
    volatile int* tq;    // TILE_Q slots: tile index, or -1 when the CTA has no more tiles
    int* tab;  // [cum (E+1) | first (E) | count (E)]
};

__device__ __forceinline__ Smem carve_smem(uint8_t* raw) {
    Smem sm;
    const uint32_t a = smem_u32(raw);
    uint8_t* base = raw + (((a + 1023u) & ~1023u) - a);
    sm.stages = base;
    sm.epi = base + STAGES * STAGE_BYTES;
    uint8_t* misc = sm.epi + EPI_BYTES;
    sm.full = reinterpret_cast<uint64_t*>(misc);
    sm.empty = sm.full + STAGES;
    sm.acc_full = sm.empty + STAGES;
    sm.acc_empty = sm.acc_full + 2;
    sm.drain = sm.acc_empty + 2;
    sm.cbar = sm.drain + 1;
    sm.tq_full = sm.cbar + COPY_NBUF;
    sm.tq_empty = sm.tq_full + TILE_Q;
    sm.tmem_base = reinterpret_cast<uint32_t*>(sm.tq_empty + TILE_Q);
    sm.abort = reinterpret_cast<volatile int*>(sm.tmem_base + 1);
    sm.tq = sm.abort + 1;
    sm.tab = const_cast<int*>(sm.tq + TILE_Q);
    return sm;
}

// Tile hand-out. Each producer CTA's TMA thread takes its first tile statically (blockIdx.x) and
// every further one from a per-GEMM counter in the plan's meta words when it has issued the loads
// of the previous one, so tiles go to whichever CTA is free first and a CTA slowed down (a tile whose
// expert weights came from DRAM rather than L2) takes fewer of them. Which CTA computes a tile does
// not change its result. The index reaches the UMMA issuer and the epilogue warps through a ring of
// TILE_Q shared-memory slots (tq_full / tq_empty); -1 ends the CTA's tiles.
constexpr int TILE_ABORT = -2;

// One thread: the j-th tile index of this CTA from the hand-out ring (TILE_ABORT if the wait ran out).
__device__ __forceinline__ int tile_take(const Smem& sm, int j, unsigned long long tmo) {
    const int slot = j % TILE_Q;
    if (!mbar_wait(&sm.tq_full[slot], (uint32_t)(j / TILE_Q) & 1u, tmo, sm.abort)) return TILE_ABORT;
    const int t = sm.tq[slot];
    mbar_arrive(&sm.tq_empty[slot]);
    return t;
}

// One GEMM tile as one CTA sees it: 128 rows of the expert-compact layout from `row` on (-1: this
// CTA of a pair has no rows in the tile), N tile n, expert e, and the work item's index in its list.
// Both GEMMs take the same items, 128 compact rows of one expert; the SwiGLU GEMM stores its rows
// in the compact layout, the down-projection's epilogue sends each row to its owner-aligned row.
struct TileRef {
    int row, n, e, item;
};

__device__ __forceinline__ TileRef tile_ref(int row, int n, int e, int item) {
    TileRef r;
    r.row = row;
    r.n = n;
    r.e = e;
    r.item = item;
    return r;
}

// SwiGLU GEMM order: expert-major; inside an expert, N tiles outer and work items inner, so the
// CTAs working at the same time share each weight tile through L2.
// tab = [cum (E+1) | first item (E) | items (E)]; items = (first compact row, expert)
__device__ __forceinline__ TileRef decode_up(int t, const int* tab, int E, const int32_t* items) {
    const int* cum = tab;
    const int* first = tab + (E + 1);
    const int* count = first + E;
    int lo = 0, hi = E - 1;  // largest e with cum[e] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int e = lo, local = t - cum[e], cnt = count[e];
    const int n = local / cnt, it = first[e] + local % cnt;
    return tile_ref(items[2 * it], n, e, it);
}

// Down-projection order: work items in hand-out order (experts by rank, each expert's items in
// compact-row order, which follows its bands in hand-out order), all N tiles of an item together.
__device__ __forceinline__ TileRef decode_down(int t, int nN, const int32_t* items) {
    const int it = t / nN;
    return tile_ref(items[2 * it], t - it * nN, items[2 * it + 1], it);
}

// One epilogue warp's staging in shared memory: two 32-row x 32-column bf16 chunk buffers, used
// alternately. put(): each lane writes its row (16-byte pieces in a lane-rotated order, free of
// bank conflicts), then lane 0 stores the chunk with one TMA tensor store.
struct EpiStage {
    uint8_t* buf;
    int eb;
    __device__ __forceinline__ void put(const CUtensorMap* tm, const uint32_t (&pk)[16], int x, int y, int lane) {
        if (lane == 0) bulk_wait_read_1();  // the store that last used this buffer has read it
        __syncwarp();
        uint4* dst = reinterpret_cast<uint4*>(buf + eb * EPI_CHUNK_BYTES + lane * (EPI_CHUNK * 2));
        const uint4 u0 = make_uint4(pk[0], pk[1], pk[2], pk[3]), u1 = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        const uint4 u2 = make_uint4(pk[8], pk[9], pk[10], pk[11]);
        const uint4 u3 = make_uint4(pk[12], pk[13], pk[14], pk[15]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int pi = (i + lane) & 3;
            dst[pi] = pi == 0 ? u0 : pi == 1 ? u1 : pi == 2 ? u2 : u3;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tm, buf + eb * EPI_CHUNK_BYTES, x, y);
            bulk_commit();
        }
        eb ^= 1;
    }
    // The same staging, then the warp stores the chunk row by row with 16-byte stores, eight rows
    // of 64 bytes per instruction: row r of the chunk to rp[i] + col_bytes, where rp[i] (i = r / 8)
    // is that row's destination as lane (lane / 4 + 8 i) holds it (nullptr: the row goes nowhere).
    __device__ __forceinline__ void put_rows(const uint32_t (&pk)[16], uint8_t* const (&rp)[4], int col_bytes,
                                             int lane) {
        // every tensor store has read its buffer: this path commits no bulk group of its own, so the
        // last group may be the one that read this buffer (put() followed by put_rows() twice)
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        uint8_t* chunk = buf + eb * EPI_CHUNK_BYTES;
        uint4* row = reinterpret_cast<uint4*>(chunk + lane * (EPI_CHUNK * 2));
        const uint4 u0 = make_uint4(pk[0], pk[1], pk[2], pk[3]), u1 = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        const uint4 u2 = make_uint4(pk[8], pk[9], pk[10], pk[11]);
        const uint4 u3 = make_uint4(pk[12], pk[13], pk[14], pk[15]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int pi = (i + lane) & 3;
            row[pi] = pi == 0 ? u0 : pi == 1 ? u1 : pi == 2 ? u2 : u3;
        }
        __syncwarp();
        const uint4* src = reinterpret_cast<const uint4*>(chunk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int piece = lane + 32 * i;  // row piece >> 2, 16-byte piece piece & 3 of its 64 bytes
            if (rp[i]) *reinterpret_cast<uint4*>(rp[i] + col_bytes + (piece & 3) * 16) = src[piece];
        }
        __syncwarp();  // the buffer is read before it is written again
        eb ^= 1;
    }
};

// Epilogue of one warp's 32 accumulator lanes of a finished SwiGLU tile at TMEM address tb (tile
// rows y..y+31 of the compact layout): columns 0-127 hold the gate and 128-255 the up projection of
// output columns n*128..; h = silu(gate) * up, rounded to bf16. An inactive warp (a pair CTA
// without rows) stores nothing.
__device__ __forceinline__ void epilogue_swiglu(EpiStage& es, const CUtensorMap* tmOut, uint32_t tb, int n, int y,
                                                bool active, int lane) {
#pragma unroll 1
    for (int c = 0; c < BN1 / 32; ++c) {
        uint32_t g[32], u[32];
        tmem_ld32(tb + c * 32, g);
        tmem_ld32(tb + BN1 + c * 32, u);
        if (active) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
                const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * __uint_as_float(u[2 * i]);
                const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * __uint_as_float(u[2 * i + 1]);
                pk[i] = pack_bf16x2(h0, h1);
            }
            es.put(tmOut, pk, n * BN1 + c * 32, y, lane);
        }
    }
}

// Where one row of a down-projection tile goes: the compact row's output row in Yp (the plan's yrow
// table, written by the permute), or, when its band is returned by the epilogue itself
// (MOE_DIRECT_TAIL: the item holding the band's last row is at or past direct_from), its row in the
// owner's slice of Ret. A padding row goes nowhere (band -1). A row whose table entries are out of
// range is reported (ST_BAD_PLAN, detail -2) and not stored.
struct DownRow {
    uint8_t* dst;  // row start, or nullptr
    int y;         // Yp row (-1: none)
    int band;      // -1: none
    bool direct;
};

__device__ __forceinline__ DownRow down_row(const Shape& s, const PlanPtrs& p, int c, int MT, int direct_from) {
    DownRow r{nullptr, -1, -1, false};
    const int y = (c >= 0 && c < s.PC_max) ? p.yrow[c] : -1;
    if (y < 0) return r;
    const int m = y / s.tbM, rb = y - m * s.tbM;
    const size_t pitch = (size_t)s.d * 2;
    if (y >= s.P_max || m >= MT || rb >= p.tiles[4 * m + 3]) {
        set_status(p.meta, ST_BAD_PLAN, -2);
        return r;
    }
    if (p.band_item[m] >= direct_from) {
        const int ret = p.tile_ret[m] + rb;
        if (ret < 0 || ret >= s.T * s.k) {
            set_status(p.meta, ST_BAD_PLAN, -2);
            return r;
        }
        r.dst = reinterpret_cast<uint8_t*>(p.Ret) + (size_t)ret * pitch;
        r.direct = true;
    } else {
        r.dst = reinterpret_cast<uint8_t*>(p.Yp) + (size_t)y * pitch;
    }
    r.y = y;
    r.band = m;
    return r;
}

// Epilogue of one warp's 32 accumulator lanes of a finished down-projection tile (BN columns of
// output columns n*BN..), rounded to bf16; lane i's row goes to dr.dst. When the warp's 32 rows are
// 32 consecutive Yp rows from y0 (a quarter of a full band: the common case), each 32-column chunk
// leaves with one TMA tensor store, else with row-by-row 16-byte stores (put_rows).
__device__ __forceinline__ void epilogue_down(EpiStage& es, const CUtensorMap* tmOut, uint32_t tb, int n, int BN,
                                              const DownRow& dr, int lane) {
    if (!__any_sync(0xffffffffu, dr.dst != nullptr)) return;  // padding rows only
    const int y0 = __shfl_sync(0xffffffffu, dr.y, 0);
    const bool tma = __all_sync(0xffffffffu, dr.dst != nullptr && !dr.direct && dr.y == y0 + lane);
    uint8_t* rp[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        rp[i] = reinterpret_cast<uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dr.dst), (lane >> 2) + 8 * i));
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tb + c * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        if (tma) es.put(tmOut, pk, n * BN + c * 32, y0, lane);
        else es.put_rows(pk, rp, (n * BN + c * 32) * 2, lane);
    }
}

// Publish one warp's rows of a finished down-projection tile (overlapped runs): the tensor stores
// lane 0 issued have completed, the row stores of every lane are ordered before lane 0 by the warp
// barrier, the async proxy is fenced against the generic one; then lane 0 adds, for each band among
// the warp's rows, that band's row count to the tile flag (ready at the band's valid rows) and to the
// band counter (ready at valid rows x N tiles), each with release semantics. The add that completes
// a band (acquire-release: it reads every other warp's released add, so their rows are ordered
// before it) stamps the trace and, for moe_forward_dma, writes the band's host record.
__device__ __forceinline__ void publish_rows(const Shape& s, const PlanPtrs& p, const DownRow& dr, int n, int lane) {
    const unsigned same = __match_any_sync(0xffffffffu, dr.band);
    unsigned leaders = __ballot_sync(0xffffffffu, dr.band >= 0 && (same & ((1u << lane) - 1u)) == 0u);
    if (!leaders) return;
    if (lane == 0) {
        bulk_wait_all();
        fence_proxy_async_global();
        __threadfence();
    }
    const uint32_t nN = (uint32_t)s.n_tiles_n2;
    for (; leaders; leaders &= leaders - 1u) {
        const int l = __ffs(leaders) - 1;
        const int m = __shfl_sync(0xffffffffu, dr.band, l);
        const uint32_t cnt = (uint32_t)__popc(__shfl_sync(0xffffffffu, same, l));
        const bool direct = __shfl_sync(0xffffffffu, dr.direct ? 1 : 0, l) != 0;  // a property of the band
        if (lane == 0) {
            red_release_gpu_add(p.flags + (size_t)m * nN + n, cnt);
            const uint32_t before = atom_acq_rel_gpu_add(p.bands + m, cnt);
            if (before + cnt == (uint32_t)p.tiles[4 * m + 3] * nN) {
                atomicMax(&p.trace[MOE_TRACE_BAND_DONE], globaltimer());
                if (p.host_rec) host_band_record(s, p, m, direct);  // the band's last rows
            }
        }
    }
    __syncwarp();
}

// Fused dispatch (MOE_FUSED_DISPATCH), the permute's row copies inside the SwiGLU GEMM: before its
// first tile, every epilogue warp of every CTA (idle until the first accumulator is ready) takes
// blocks of DISPATCH_ROWS compact rows from a queue in row order, i.e. expert by expert, copies each
// row's token (or zeros for a padding row) into Xc with 16-byte loads and stores, and then adds the
// block's rows to its expert's count with release semantics. A TMA thread loads an expert's rows
// only once that count covers every row of the expert (acquire, then an async-proxy fence). The
// copying warps wait on nothing, so every count completes whatever CTAs are resident.
constexpr int DISPATCH_ROWS = 4;

__device__ void dispatch_rows(const Shape& s, const PlanPtrs& p) {
    const int lane = threadIdx.x & 31;
    int PC = p.meta[META_PC];
    if (PC < 0 || PC > s.PC_max) PC = 0;
    const int nb = PC / DISPATCH_ROWS;  // PC is a multiple of 128
    const int vec = s.d / 8;            // 16-byte vectors per row
    const uint4* xs = reinterpret_cast<const uint4*>(p.x);
    uint4* xc = reinterpret_cast<uint4*>(p.Xc);
    constexpr int V = 16;               // vectors per lane in flight
    for (;;) {
        int b = 0;
        if (lane == 0) b = atomicAdd(&p.meta[META_DISPATCH], 1);
        b = __shfl_sync(0xffffffffu, b, 0);
        if (b >= nb) break;
        const int r0 = b * DISPATCH_ROWS;
        const int e = p.items_up[2 * (r0 / BM) + 1];  // a block lies in one 128-row item of one expert
        int tk = (lane < DISPATCH_ROWS) ? p.tok_of[r0 + lane] : -1;
        const bool bad = __any_sync(0xffffffffu, tk < -1 || tk >= s.T) || e < 0 || e >= s.E;
        if (bad) {
            if (lane == 0) set_status(p.meta, ST_BAD_PLAN, -4);
            break;
        }
        for (int r = 0; r < DISPATCH_ROWS; ++r) {
            const int t = __shfl_sync(0xffffffffu, tk, r);
            uint4* dst = xc + (size_t)(r0 + r) * vec;
            for (int base = 0; base < vec; base += 32 * V) {
                uint4 v[V];
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    const int vi = base + i * 32 + lane;
                    v[i] = make_uint4(0, 0, 0, 0);
                    if (t >= 0 && vi < vec) v[i] = __ldg(xs + (size_t)t * vec + vi);
                }
#pragma unroll
                for (int i = 0; i < V; ++i) {
                    const int vi = base + i * 32 + lane;
                    if (vi < vec) dst[vi] = v[i];
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence();
            red_release_gpu_add(p.xrows + e, DISPATCH_ROWS);
        }
    }
    __syncwarp();
}

// TMA thread of a SwiGLU GEMM with fused dispatch: wait (bounded) until every compact row of expert e
// has been copied, then order the async-proxy loads after the acquire. Returns false on timeout.
__device__ __forceinline__ bool wait_expert_rows(const Shape& s, const PlanPtrs& p, int e, volatile int* abort,
                                                 int where) {
    const uint32_t need = (uint32_t)p.experts[8 * e + 4] * BM;
    if (ld_acquire_gpu(p.xrows + e) < need) {
        const unsigned long long t0 = globaltimer();
        while (ld_acquire_gpu(p.xrows + e) < need) {
            if (*abort) return false;
            if (globaltimer() - t0 > s.timeout_ns) {
                set_status(p.meta, ST_PIPE_TIMEOUT, where);
                return false;
            }
            __nanosleep(64);
        }
    }
    fence_proxy_async_global();
    return true;
}

// Bounds check of the plan entries a GEMM launch reads, by all threads of a CTA before any tile:
// work items (first compact row, expert) and the expert table of the item list. Returns nonzero if
// this thread found a bad entry. Every CTA reaches the same answer, so a corrupt plan stops the whole
// launch; the status detail is -1 (SwiGLU items) or -2 (down-projection items). The entries a
// down-projection row is sent by (yrow, the band tables) are checked row by row (down_row).
__device__ __forceinline__ int plan_items_bad(const Shape& s, const PlanPtrs& p, int mode, int NI) {
    int bad = 0;
    const int32_t* items = (mode == 1) ? p.items_up : p.items_down;
    for (int it = threadIdx.x; it < NI && !bad; it += blockDim.x) {
        const int crow = items[2 * it], e = items[2 * it + 1];
        if (e < 0 || e >= s.E || crow < 0 || crow % BM != 0 || crow + BM > s.PC_max) bad = it + 1;
    }
    for (int e = threadIdx.x; e < s.E && !bad; e += blockDim.x) {
        const int cnt = p.experts[8 * e + 4], first = p.experts[8 * e + ((mode == 1) ? 5 : 6)];
        if (cnt < 0 || first < 0 || first + cnt > NI) bad = NI + e + 1;
    }
    return bad;
}

template <int MODE>  // 1: SwiGLU up-projection -> Hc; 2: down-projection -> Yp (+ flags / consumer)
__global__ void __launch_bounds__(GEMM_THREADS_MAX, 1)
    gemm_kernel(Shape s, PlanPtrs p, const __grid_constant__ CUtensorMap tmA,
                const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                const __grid_constant__ CUtensorMap tmOut, int num_producers, int overlapped) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm = carve_smem(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const bool producer = (int)blockIdx.x < num_producers;

    int MT = p.meta[META_MTILES], NI = p.meta[(MODE == 1) ? META_ITEMS_UP : META_ITEMS];
    if (MT < 0 || MT > s.MT_max || NI < 0 || NI > ((MODE == 1) ? s.IU_max : MT)) MT = NI = 0;
    const int nN = (MODE == 1) ? s.ffn / BN1 : s.n_tiles_n2;
    const int BN = (MODE == 1) ? 2 * BN1 : s.bn2;  // UMMA N
    const int KB = ((MODE == 1) ? s.d : s.ffn) / BK;
    const int bad_item = __syncthreads_or(plan_items_bad(s, p, MODE, NI));
    if (bad_item) NI = 0;  // no tile runs; the copy engines stop at the abort word set below
    const int total = NI * nN;
    const uint32_t tx_bytes = A_STAGE_BYTES + BN * BK * 2;
    const unsigned long long tmo = s.timeout_ns;
    const bool dispatch = MODE == 1 && (s.flags & MOE_FUSED_DISPATCH);
    // MOE_DIRECT_TAIL: items from `direct_from` on have a tile among the last `window` hand-out
    // positions (item i's tiles are i*nN .. i*nN+nN-1), so they may complete bands in the last wave;
    // their epilogue writes those bands' rows into Ret and the copy engines skip them
    int direct_from = INT_MAX;
    if (MODE == 2 && overlapped && (s.flags & MOE_DIRECT_TAIL)) {
        const int window = s.tail_window > 0 ? s.tail_window : num_producers, thr = total - window;
        direct_from = thr <= 0 ? 0 : min(NI, thr / nN);
    }

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc_full[i], 1);
            mbar_init(&sm.acc_empty[i], 128);
        }
        mbar_init(sm.drain, 1);
        for (int i = 0; i < COPY_NBUF; ++i) mbar_init(&sm.cbar[i], 1);
        for (int i = 0; i < TILE_Q; ++i) {
            mbar_init(&sm.tq_full[i], 1);
            mbar_init(&sm.tq_empty[i], 1 + 4);
        }
        *sm.abort = bad_item ? 1 : 0;
        if (bad_item) set_status(p.meta, ST_BAD_PLAN, -MODE);
        mbar_fence_init();
    }
    if (MODE == 1) {
        for (int e = tid; e < s.E; e += blockDim.x) {
            sm.tab[(s.E + 1) + e] = p.experts[8 * e + 5];         // first work item
            sm.tab[(s.E + 1) + s.E + e] = p.experts[8 * e + 4];   // work items
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int e = 0; e < s.E; ++e) {
                sm.tab[e] = acc;
                acc += sm.tab[(s.E + 1) + s.E + e] * nN;
            }
            sm.tab[s.E] = acc;
        }
    }
    if (producer && warp == 1) {
        tmem_alloc(sm.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    if (producer && tid == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        tma_prefetch_desc(&tmOut);
        if (MODE == 1) tma_prefetch_desc(&tmB1);
        if (MODE == 2) atomicMin(&p.trace[MOE_TRACE_GEMM2_START], globaltimer());
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();  // MOE_PDL: the previous kernel's outputs (the plan tables above were complete before)
    griddep_launch();
    const ClockSpan clk = clock_span_start(blockIdx.x == 0 && tid == 0);
    const uint32_t tmem = producer ? *sm.tmem_base : 0u;
    unsigned long long last_end = 0;
    const uint32_t stall = (s.flags & MOE_TEST_STALL_CONSUMER) ? 1u : 0u;  // a count no band reaches

    // Extra warps (launched with MOE_COPY_WARPS): SIMT copy engines beside the GEMM warps.
    if (warp >= GEMM_WARPS) {
        if (MODE == 2 && overlapped) copy_units_simt(s, p, sm.abort, META_QUEUE, stall, direct_from);
        return;
    }

    if (producer) {
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer ----------------
            int st = 0;
            uint32_t ph = 0, issued = 0, last_ph = 0;
            bool ok = true;
            int t = blockIdx.x;  // first tile static, the others from the hand-out counter
            int ready_e = -1;    // fused dispatch: the expert whose rows are known to be copied
            int* tile_counter = &p.meta[(MODE == 1) ? META_TILES_UP : META_TILES_DOWN];
            const int claim_kb = KB > 8 ? KB - 8 : 0;
            for (int j = 0; ok; ++j) {
                const int slot = j % TILE_Q;
                if (!mbar_wait(&sm.tq_empty[slot], ((uint32_t)(j / TILE_Q) & 1u) ^ 1u, tmo, sm.abort)) {
                    ok = false;
                    break;
                }
                sm.tq[slot] = t < total ? t : -1;
                mbar_arrive(&sm.tq_full[slot]);
                if (t >= total) break;
                const TileRef tr = (MODE == 1) ? decode_up(t, sm.tab, s.E, p.items_up) : decode_down(t, nN, p.items_down);
                if (MODE == 1 && dispatch && tr.e != ready_e) {
                    if (!wait_expert_rows(s, p, tr.e, sm.abort, 30)) {
                        ok = false;
                        break;
                    }
                    ready_e = tr.e;
                }
                int next = total;
                for (int kb = 0; kb < KB; ++kb) {
                    // the next tile is taken a few k-blocks before this one's loads are all issued,
                    // so the atomic's latency is hidden: a CTA that ran slower (weights streamed
                    // from DRAM) takes fewer tiles
                    if (kb == claim_kb) next = num_producers + atomicAdd(tile_counter, 1);
                    if (!mbar_wait(&sm.empty[st], ph ^ 1u, tmo, sm.abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.full[st], tx_bytes);
                    uint8_t* a = sm.stages + st * STAGE_BYTES;
                    uint8_t* b = a + A_STAGE_BYTES;
                    tma_load_2d(a, &tmA, &sm.full[st], kb * BK, tr.row);  // 128 compact rows
                    if (MODE == 1) {
                        tma_load_3d(b, &tmB0, &sm.full[st], kb * BK, tr.n * BN1, tr.e);
                        tma_load_3d(b + BN1 * BK * 2, &tmB1, &sm.full[st], kb * BK, tr.n * BN1, tr.e);
                    } else {
                        tma_load_3d(b, &tmB0, &sm.full[st], kb * BK, tr.n * BN, tr.e);
                    }
                    issued |= 1u << st;
                    last_ph = (last_ph & ~(1u << st)) | (ph << st);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                t = next;
            }
            if (!ok) {
                if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 0);
                *sm.abort = 1;
                int never = 0;
                for (int i = 0; i < STAGES; ++i)  // let loads in flight land before the CTA leaves
                    if (issued & (1u << i)) mbar_wait(&sm.full[i], (last_ph >> i) & 1u, tmo, &never);
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------- UMMA issuer ----------------
            const uint32_t idesc = umma_idesc_bf16(BM, BN);
            int st = 0, b = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true, any = false;
            for (int j = 0; ok; ++j) {
                const int t = tile_take(sm, j, tmo);
                if (t == TILE_ABORT) {
                    ok = false;
                    break;
                }
                if (t < 0) break;
                if (!mbar_wait(&sm.acc_empty[b], aph ^ 1u, tmo, sm.abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + (uint32_t)(b * 256);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!mbar_wait(&sm.full[st], ph, tmo, sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sm.stages + st * STAGE_BYTES);
                    const uint64_t ad = sdesc_sw128(a_addr);
                    const uint64_t bd = sdesc_sw128(a_addr + A_STAGE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)  // +32 bytes along K per UMMA_K = 16
                        umma_bf16(dt, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    umma_commit(&sm.empty[st]);
                    any = true;
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&sm.acc_full[b]);
                b ^= 1;
                if (b == 0) aph ^= 1u;
            }
            if (!ok) {
                if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 1);
                *sm.abort = 1;
                if (any) {  // wait for the UMMAs in flight before TMEM is released
                    int never = 0;
                    umma_commit(sm.drain);
                    mbar_wait(sm.drain, 0, tmo, &never);
                }
            }
        } else if (warp >= 2) {
            // ---------------- epilogue ----------------
            // Each warp owns TMEM lanes 32q..32q+31 (tile rows). Per 32-column chunk: tcgen05.ld,
            // convert, write the 32 x 32 bf16 chunk to a shared staging buffer (each lane its row,
            // 16-byte pieces in a lane-rotated order, free of bank conflicts), then lane 0 issues one
            // TMA tensor store of the chunk. Two staging buffers per warp alternate.
            const int q = warp & 3;  // TMEM lane quarter this warp may access
            const bool flags = (MODE == 2) && overlapped;
            if (MODE == 1 && dispatch) dispatch_rows(s, p);
            EpiStage es{sm.epi + (warp - 2) * 2 * EPI_CHUNK_BYTES, 0};
            int b = 0;
            uint32_t aph = 0;
            for (int j = 0;; ++j) {
                int t = 0;
                if (lane == 0) t = tile_take(sm, j, tmo);
                t = __shfl_sync(0xffffffffu, t, 0);
                if (t == TILE_ABORT) {
                    if (lane == 0) {
                        if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 3);
                        *sm.abort = 1;
                    }
                    break;
                }
                if (t < 0) break;
                const TileRef tr = (MODE == 1) ? decode_up(t, sm.tab, s.E, p.items_up) : decode_down(t, nN, p.items_down);
                if (!mbar_wait(&sm.acc_full[b], aph, tmo, sm.abort)) {
                    if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 2);
                    *sm.abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 256);
                const int c0 = tr.row + q * 32;  // this warp's first compact row
                if (MODE == 1) {
                    epilogue_swiglu(es, &tmOut, tb, tr.n, c0, true, lane);
                    tc_fence_before();
                    mbar_arrive(&sm.acc_empty[b]);
                } else {
                    const DownRow dr = down_row(s, p, c0 + lane, MT, direct_from);
                    epilogue_down(es, &tmOut, tb, tr.n, BN, dr, lane);
                    tc_fence_before();
                    mbar_arrive(&sm.acc_empty[b]);
                    if (flags) publish_rows(s, p, dr, tr.n, lane);
                    const bool stored = __any_sync(0xffffffffu, dr.band >= 0);
                    if (lane == 0 && stored) last_end = globaltimer();
                }
                b ^= 1;
                if (b == 0) aph ^= 1u;
            }
            if (lane == 0) bulk_wait_all();  // staging buffers stay valid until every store is done
            __syncwarp();
        }
    }
    tc_fence_before();
    named_bar_sync(1, GEMM_THREADS);  // the GEMM warps only: extra copy warps run on independently
    if (producer && warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    if (MODE == 2 && producer && warp >= 2 && lane == 0 && last_end)
        atomicMax(&p.trace[MOE_TRACE_GEMM2_END], last_end);
    clock_span_add(p, clk, MODE == 2 ? MOE_TRACE_DOWN_CYCLES : MOE_TRACE_UP_CYCLES);

    if (MODE == 2 && overlapped && (!producer || (s.flags & MOE_TAIL_ASSIST)))
        copy_units(s, p, sm.stages, sm.cbar, sm.abort, META_QUEUE, true, stall, direct_from);
}

// =============================================================================================
// Expert GEMMs on CTA pairs (MOE_PAIR_UMMA). A cluster of two CTAs computes one 256-row x 256-column
// UMMA tile: each CTA stages the 128 rows of one work item of the expert and one half of the B
// tile; one thread of rank 0 issues tcgen05.mma.cta_group::2, and each CTA's TMEM receives its own
// 128 rows x 256 columns, so each CTA runs the single-CTA epilogue on its rows.
//   MODE 1 (SwiGLU up-projection): rank 0 stages the gate half of B (W1 rows), rank 1 the up half
//       (W3 rows); each CTA's accumulator holds 128 gate | 128 up columns. Work items of an expert
//       in pairs, N tiles outer.
//   MODE 2 (down-projection): rank 0 stages rows 0-127 of the 256-row W2 tile, rank 1 rows
//       128-255; each CTA's item is 128 compact rows of one expert, whose epilogue sends every row
//       to its owner-aligned band and publishes the band flags as in gemm_kernel. Work items of an
//       expert in pairs, in hand-out order, all N tiles of a pair item together. Consumer CTAs (the last
//       consumer_ctas blocks, whole clusters) and, with tail assist, finished producer CTAs run the
//       bulk copy engines.
// An expert with an odd number of work items leaves rank 1 without rows in its last pair tile: it
// still loads its B half (rank 0's columns need it), its A box lies past the last compact row
// (zeros), and its accumulator rows are not stored.
//
// Barriers: full[s] on rank 0 (the stage's bytes of both CTAs landed: rank 0 arms it with both
// CTAs' byte counts, and rank 1's TMA loads complete on it through cta_group::2), empty[s] (UMMAs
// of the stage done; committed to both CTAs), acc_full[b] (committed to both CTAs), acc_empty[b]
// on rank 0 (count 8: the four epilogue warps of each CTA). Every wait is bounded; a timeout
// raises the abort word of both CTAs.
//
// Tile hand-out: rank 0's TMA thread takes every tile of the pair from the GEMM's counter in the
// plan's meta words (the next one a few k-blocks before the current one's loads are all issued), so
// tiles go to whichever pair is free first and no tile waits for a particular pair to be resident.
// It publishes each index in a ring of PAIR_TILE_Q slots of both CTAs: its own slot with a store and
// an arrive on tq_full, the peer's with st.async, which completes 4 transaction bytes on the peer's
// tq_full (armed by the peer's TMA thread, once at start and again each time it has read the slot).
// Rank 0's tq_empty (count 5) collects rank 0's UMMA issuer and epilogue warps. Rank 1's readers
// need no arrive there. Its TMA thread: rank 0's TMA thread cannot run more than PAIR_STAGES k-blocks
// ahead of it (every stage's barrier waits for rank 1's loads), so when rank 0 reuses a slot
// PAIR_TILE_Q tiles later, rank 1 has long since read it. Its epilogue warps: rank 0's TMA thread
// writes the slot of its tile j + 8 only after issuing every k-block of tile j + 7, which needs the
// stages freed by the UMMAs of a k-block of tile j + 8 - ceil(7 / KB) or later, whose tile began only
// after both CTAs' epilogues released the accumulator of tile j + 6 - ceil(7 / KB) >= j + 2 (KB >= 2
// k-blocks per tile: d, ffn >= 128); the epilogue takes its tiles in order, so it read slot j before.
// (A cluster-scope arrive waits for the SM's outstanding memory operations: four of them per tile
// held rank 1's epilogue up on short tiles.)
// =============================================================================================
struct PairSmem {
    uint8_t* stages;
    uint8_t* epi;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    uint64_t* tq_full;   // PAIR_TILE_Q tile hand-out slots (see above)
    uint64_t* tq_empty;
    uint64_t* cbar;      // copy engines (down-projection consumers and tail assist)
    uint32_t* tmem_base;
    uint32_t* peer_base;
    volatile uint32_t* peer_k;  // rank 0: k-blocks rank 1's TMA thread issued (abort path)
    volatile int* abort;
    volatile int* tq;
    volatile int* nprod;  // producer CTAs of this launch (the launch's, or MOE_ADAPTIVE_CONSUMERS')
    int* tab;  // [cum (E+1) | first item (E) | items (E) | first direct item]
};

__device__ __forceinline__ PairSmem carve_pair(uint8_t* raw) {
    PairSmem sm;
    const uint32_t a = smem_u32(raw);
    uint8_t* base = raw + (((a + 1023u) & ~1023u) - a);
    sm.stages = base;
    sm.epi = base + PAIR_STAGES * PAIR_STAGE_BYTES;
    uint8_t* misc = sm.epi + EPI_BYTES;
    sm.full = reinterpret_cast<uint64_t*>(misc);
    sm.empty = sm.full + PAIR_STAGES;
    sm.acc_full = sm.empty + PAIR_STAGES;
    sm.acc_empty = sm.acc_full + 2;
    sm.drain = sm.acc_empty + 2;
    sm.tq_full = sm.drain + 1;
    sm.tq_empty = sm.tq_full + PAIR_TILE_Q;
    sm.cbar = sm.tq_empty + PAIR_TILE_Q;
    sm.tmem_base = reinterpret_cast<uint32_t*>(sm.cbar + COPY_NBUF);
    sm.peer_base = sm.tmem_base + 1;
    sm.peer_k = sm.peer_base + 1;
    sm.abort = reinterpret_cast<volatile int*>(const_cast<uint32_t*>(sm.peer_k) + 1);
    sm.tq = sm.abort + 1;
    sm.nprod = sm.tq + PAIR_TILE_Q;
    sm.tab = const_cast<int*>(sm.nprod + 1);
    return sm;
}
static_assert(COPY_NBUF * COPY_PIECE <= PAIR_STAGES * PAIR_STAGE_BYTES, "copy staging must fit the pair stage area");

// One thread: the j-th tile index of the pair from this CTA's hand-out ring (TILE_ABORT if the wait
// ran out). Rank 1's slots are filled by st.async from rank 0, so the wait acquires at cluster
// scope. The caller then releases the slot: rank 0's consumers with a local arrive on tq_empty, rank
// 1's epilogue warps with a cluster arrive on rank 0's tq_empty, rank 1's TMA thread by arming its
// tq_full for the slot's next use.
__device__ __forceinline__ int pair_tile_wait(const PairSmem& sm, int j, unsigned long long tmo) {
    const int slot = j % PAIR_TILE_Q;
    if (!mbar_wait_cluster(&sm.tq_full[slot], (uint32_t)(j / PAIR_TILE_Q) & 1u, tmo, sm.abort)) return TILE_ABORT;
    return sm.tq[slot];
}

// Raise the abort word of both CTAs of the pair.
__device__ __forceinline__ void pair_abort(const PairSmem& sm, uint32_t rank) {
    *sm.abort = 1;
    st_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(sm.abort)), rank ^ 1u), 1u);
}

// Abort path of a pair (rank 0's TMA thread, after both CTAs have stopped issuing): no TMA load of the
// pair may still be in flight when either CTA leaves. Both TMA threads walk the same sequence of
// k-blocks (stage i % PAIR_STAGES, phase (i / PAIR_STAGES) & 1): rank 0 arms k-block i's full
// barrier with both CTAs' bytes and issues its own loads, rank 1's loads complete on that barrier.
// `a` k-blocks were armed and loaded by rank 0, `b` loaded by rank 1; the two differ by at most
// PAIR_STAGES, and every k-block below min(a, b) got both. For i in [b, a) rank 1's bytes never come:
// they are completed without a copy; for i in [a, b) rank 0 never armed the phase: it arrives now,
// expecting rank 1's bytes. Then every barrier's last phase is waited for (bounded): a phase completes
// only when all of its loads have landed, and earlier phases completed before it.
__device__ __forceinline__ void pair_settle(const PairSmem& sm, uint32_t a, uint32_t b, unsigned long long tmo) {
    const uint32_t peer_bytes = PAIR_A_BYTES + PAIR_B_BYTES;  // rank 1's loads of one k-block
    const uint32_t lo = a < b ? a : b, hi = a < b ? b : a;
    for (uint32_t i = lo; i < hi; ++i) {
        uint64_t* bar = &sm.full[i % PAIR_STAGES];
        if (i < a) mbar_complete_tx(bar, peer_bytes);
        else mbar_arrive_expect_tx(bar, peer_bytes);
    }
    int never = 0;
    for (uint32_t i = hi > (uint32_t)PAIR_STAGES ? hi - PAIR_STAGES : 0u; i < hi; ++i)
        mbar_wait(&sm.full[i % PAIR_STAGES], (i / PAIR_STAGES) & 1u, tmo, &never);
}

// Largest e with cum[e] <= t (cum non-decreasing, cum[0] = 0 <= t).
__device__ __forceinline__ int tab_segment(const int* cum, int E, int t) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Pair tile t -> this CTA's rows (SwiGLU tiles). Order as in decode_up with two work items per pair:
// the table's experts in order (ids in `eid`, or the table's order is the id order when eid is
// null), N tiles outer, pairs inner; rank r takes item 2 * pair + r of the expert (row -1: none).
__device__ __forceinline__ TileRef decode_pair_up(int t, const int* tab, int E, const int32_t* items,
                                                  uint32_t rank, const int* eid = nullptr) {
    const int* cum = tab;
    const int* first = tab + (E + 1);
    const int* count = first + E;
    const int r = tab_segment(cum, E, t), local = t - cum[r], cnt = count[r], np = (cnt + 1) >> 1;
    const int e = eid ? eid[r] : r;
    const int n = local / np, it = 2 * (local - n * np) + (int)rank;
    if (it >= cnt) return tile_ref(-1, n, e, -1);
    const int item = first[r] + it;
    return tile_ref(items[2 * item], n, e, item);
}

// Pair tile t -> this CTA's rows (down-projection tiles). tab lists the experts in hand-out order
// (first down-projection item, items); the expert's items in pairs, all nN tiles of a pair item
// together (item first), or, for an expert of at most n_outer_items items, one N tile of all its
// pair items after another, except for the last expert, whose bands then still complete one after
// another while its tiles run; rank r takes item 2 * pair + r (row -1: none, with the expert of
// rank 0's item).
__device__ __forceinline__ TileRef decode_pair_down(int t, const int* tab, int E, int nN, const int32_t* items,
                                                    uint32_t rank, int n_outer_items) {
    const int* cum = tab;
    const int* first = tab + (E + 1);
    const int* count = first + E;
    const int r = tab_segment(cum, E, t), local = t - cum[r];
    int pi, n;
    if (count[r] <= n_outer_items && cum[r + 1] != cum[E]) {  // the last expert's tiles stay item first
        const int np = (count[r] + 1) >> 1;  // >= 1: an expert without items owns no tile
        n = local / np;
        pi = local - n * np;
    } else {
        pi = local / nN;
        n = local - pi * nN;
    }
    const int it = 2 * pi + (int)rank;
    if (it >= count[r]) return tile_ref(-1, n, items[2 * (first[r] + 2 * pi) + 1], -1);
    const int item = first[r] + it;
    return tile_ref(items[2 * item], n, items[2 * item + 1], item);
}

// The CTA-pair GEMM. MODE 1: SwiGLU tiles -> Hc; 2: down-projection tiles -> Yp (+ flags, consumer
// CTAs); 3: both in one launch (MOE_FUSED_GEMMS). In MODE 3 the SwiGLU tiles are handed out first,
// experts in hand-out order (the most loaded first); each SwiGLU epilogue warp, once its TMA stores
// have completed, fences the async proxy and release-adds 1 to its expert's count (xready), and a
// TMA thread starts an expert's down-projection tiles only when that count covers every SwiGLU tile
// quarter of the expert (acquire, then an async-proxy fence before the loads of Hc). So the
// down-projection starts on the SMs that finish their SwiGLU tiles instead of after the whole GEMM;
// the consumer clusters take SwiGLU tiles too and start copying when those run out. Every count is
// completed by epilogue warps that wait on nothing of the down-projection, so no wait can stall for
// good. Operands: mA / mB0 / mB1 / mOut are the launch's (MODE 1: Xc, W1, W3, Hc store; MODE 2: Hc,
// W2 halves twice, Yp store); MODE 3 passes the SwiGLU ones there and the down-projection's as
// mA2 / mB2 / mOut2.
template <int MODE>
__device__ __forceinline__ void pair_body(const Shape& s, const PlanPtrs& p, const CUtensorMap* mA,
                                          const CUtensorMap* mB0, const CUtensorMap* mB1, const CUtensorMap* mOut,
                                          const CUtensorMap* mA2, const CUtensorMap* mB2, const CUtensorMap* mOut2,
                                          int num_producers, int overlapped) {
    constexpr bool HAS_UP = MODE != 2, HAS_DN = MODE != 1, FUSED = MODE == 3;
    extern __shared__ uint8_t smem_raw[];
    const PairSmem sm = carve_pair(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int E = s.E;
    int MT = HAS_DN ? p.meta[META_MTILES] : 0;
    int NU = HAS_UP ? p.meta[META_ITEMS_UP] : 0;
    int ND = HAS_DN ? p.meta[META_ITEMS] : 0;
    if (MT < 0 || MT > s.MT_max || NU < 0 || NU > s.IU_max || ND < 0 || ND > MT) MT = NU = ND = 0;
    const int nN_up = s.ffn / BN1, nN_dn = s.n_tiles_n2;
    const int KB_up = s.d / BK, KB_dn = s.ffn / BK;
    const unsigned long long tmo = s.timeout_ns;
    const bool dispatch = HAS_UP && (s.flags & MOE_FUSED_DISPATCH);
    const int bad_item = __syncthreads_or((HAS_UP ? plan_items_bad(s, p, 1, NU) : 0) |
                                          (HAS_DN ? plan_items_bad(s, p, 2, ND) : 0));  // same in every CTA
    if (bad_item) NU = ND = 0;
    // expert tables: the down-projection's at tab ([cum (E+1) | first item (E) | items (E) | first
    // direct item]); the SwiGLU one at tab in MODE 1, after the down-projection's in MODE 3 (with the
    // experts' ids, as its experts are in hand-out order), then the SwiGLU tile quarters per expert
    int* const tab_up = sm.tab + (FUSED ? 3 * E + 2 : 0);
    int* const eid_up = tab_up + 3 * E + 1;
    int* const xexp = eid_up + E;

    if (tid == 0) {
        for (int i = 0; i < PAIR_STAGES; ++i) {
            mbar_init(&sm.full[i], 1);
            mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.acc_full[i], 1);
            mbar_init(&sm.acc_empty[i], 8);
        }
        mbar_init(sm.drain, 1);
        for (int i = 0; i < PAIR_TILE_Q; ++i) {
            mbar_init(&sm.tq_full[i], 1);
            mbar_init(&sm.tq_empty[i], 1 + 4);
        }
        for (int i = 0; i < COPY_NBUF; ++i) mbar_init(&sm.cbar[i], 1);
        *sm.abort = bad_item ? 1 : 0;  // a corrupt plan also stops the copy engines
        if (bad_item && rank == 0) set_status(p.meta, ST_BAD_PLAN, -MODE);
        mbar_fence_init();
        if (rank == 1)  // arm every slot for rank 0's first st.async
            for (int i = 0; i < PAIR_TILE_Q; ++i) mbar_arrive_expect_tx(&sm.tq_full[i], 4);
    }
    if (MODE == 1) {
        for (int e = tid; e < E; e += blockDim.x) {
            sm.tab[(E + 1) + e] = p.experts[8 * e + 5];         // first work item
            sm.tab[(E + 1) + E + e] = p.experts[8 * e + 4];     // work items
        }
        __syncthreads();
        if (tid == 0) {
            int acc = 0;
            for (int e = 0; e < E; ++e) {
                sm.tab[e] = acc;
                acc += ((sm.tab[(E + 1) + E + e] + 1) >> 1) * nN_up;
            }
            sm.tab[E] = acc;
        }
    } else if (tid == 0) {
        // experts in hand-out order: each expert's down-projection items are contiguous in the item
        // list, experts in hand-out order, so sorting the first items (0 <= first <= ND, checked by
        // plan_items_bad) gives the order and the item counts
        int* first = sm.tab + (E + 1);
        int* count = first + E;
        for (int e = 0; e < E; ++e) {
            const int f = p.experts[8 * e + 6];
            int i = e;
            while (i > 0 && first[i - 1] > f) {
                first[i] = first[i - 1];
                --i;
            }
            first[i] = f;
        }
        int acc = 0;
        for (int r = 0; r < E; ++r) {
            count[r] = ((r + 1 < E) ? first[r + 1] : ND) - first[r];
            sm.tab[r] = acc;
            acc += ((count[r] + 1) >> 1) * nN_dn;
        }
        sm.tab[E] = acc;
        // MOE_ADAPTIVE_CONSUMERS: the tiles are of one size and handed out as pairs become free, so
        // the down-projection takes ceil(tiles / producer pairs) waves. The fewest waves any
        // partition with at least one consumer pair allows is w = ceil(tiles / (pairs - 1)); the
        // fewest producer pairs that still finish in w waves is ceil(tiles / w), and every other
        // pair copies. (With the launch's fixed partition one pair too few costs a whole extra
        // wave of tiles when the tile count lies just above a multiple of the producer pairs.)
        int prod = num_producers;
        const int pairs = (int)gridDim.x / 2;
        if (overlapped && (s.flags & MOE_ADAPTIVE_CONSUMERS) && acc > 0 && pairs >= 2) {
            const int w = (acc + pairs - 2) / (pairs - 1);
            prod = 2 * ((acc + w - 1) / w);
        }
        *sm.nprod = prod;
        if (blockIdx.x == 0 && overlapped) p.meta[META_PRODUCERS] = prod;
        // MOE_DIRECT_TAIL: the first item of the first pair item with a tile among the last `window`
        // hand-out positions, i.e. whose last tile is (the pair items' last tiles rise with the item
        // index, so every later item has one there too): those items may complete bands in the last
        // wave, so their epilogue and every later one's write those bands into Ret. In the first
        // expert that reaches the window (rel = the window's start inside its tiles) that is pair
        // item rel / nN (item first: pair item p's tiles end at (p + 1) nN - 1) or
        // rel - (nN - 1) np (N tile by N tile: pair item p's last tile is at (nN - 1) np + p)
        int from = INT_MAX;
        if (overlapped && (s.flags & MOE_DIRECT_TAIL) && ND > 0 && acc > 0) {
            const int window = s.tail_window > 0 ? s.tail_window : prod / 2, thr = acc - window;
            from = ND;
            for (int r = 0; r < E; ++r) {
                const int np = (count[r] + 1) >> 1;
                if (np == 0 || sm.tab[r + 1] <= thr) continue;
                const bool n_outer = count[r] <= s.down_n_outer_items && sm.tab[r + 1] != acc;
                const int rel = thr - sm.tab[r];
                const int pi = rel <= 0 ? 0 : (n_outer ? max(0, rel - (nN_dn - 1) * np) : rel / nN_dn);
                if (pi < np) {
                    from = first[r] + 2 * pi;
                    break;
                }
            }
        }
        sm.tab[3 * E + 1] = from;
        if (FUSED) {
            // SwiGLU table, experts in hand-out rank order (a permutation: the plan's ranks)
            int* ufirst = tab_up + (E + 1);
            int* ucount = ufirst + E;
            for (int e = 0; e < E; ++e) {
                const int r = min(max(p.experts[8 * e + 3], 0), E - 1);
                ufirst[r] = p.experts[8 * e + 5];
                ucount[r] = p.experts[8 * e + 4];
                eid_up[r] = e;
                xexp[e] = ((p.experts[8 * e + 4] + 1) >> 1) * nN_up * 8;  // epilogue warps of both CTAs
            }
            int uacc = 0;
            for (int r = 0; r < E; ++r) {
                tab_up[r] = uacc;
                uacc += ((ucount[r] + 1) >> 1) * nN_up;
            }
            tab_up[E] = uacc;
        }
    }
    if (MODE == 1 && tid == 0) *sm.nprod = num_producers;
    __syncthreads();
    const int num_prod = *sm.nprod;
    const bool producer = (int)blockIdx.x < num_prod;  // even: both CTAs of a cluster share the role
    const bool gemm_cta = producer || FUSED;            // fused: consumer clusters take SwiGLU tiles
    if (gemm_cta && warp == 1) {
        __syncwarp();
        tmem_alloc_pair(sm.tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (tid == 0) {
        tma_prefetch_desc(mA);
        tma_prefetch_desc(mB0);
        tma_prefetch_desc(mB1);
        tma_prefetch_desc(mOut);
        if (FUSED) {
            tma_prefetch_desc(mA2);
            tma_prefetch_desc(mB2);
            tma_prefetch_desc(mOut2);
        }
        if (MODE == 2 && producer) atomicMin(&p.trace[MOE_TRACE_GEMM2_START], globaltimer());
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs started, their barriers initialised and TMEM allocated
    tc_fence_after();
    if (gemm_cta && rank == 1 && tid == 0) st_cluster_u32(mapa_shared(smem_u32(sm.peer_base), 0u), *sm.tmem_base);
    cluster_sync();  // rank 1's column base delivered to rank 0
    // MOE_PDL: this launch may have started while the previous kernel was finishing; wait for its
    // outputs here. The plan tables read above were complete before that kernel started.
    griddep_wait();
    griddep_launch();
    const ClockSpan clk = clock_span_start(blockIdx.x == 0 && tid == 0);
    const uint32_t tmem = gemm_cta ? *sm.tmem_base : 0u;
    const int N_up = HAS_UP ? ((NU > 0 && tab_up[E] > 0) ? tab_up[E] : 0) : 0;  // SwiGLU pair tiles
    const int N_dn = HAS_DN ? ((ND > 0 && sm.tab[E] > 0) ? sm.tab[E] : 0) : 0;  // down-projection pair tiles
    const int total = N_up + N_dn;  // tile t: [0, N_up) SwiGLU, [N_up, total) down-projection
    const bool bad = gemm_cta && rank == 0 && *sm.peer_base != tmem;  // not one pair allocation
    const uint32_t stall = (s.flags & MOE_TEST_STALL_CONSUMER) ? 1u : 0u;  // a count no band reaches
    unsigned long long last_end = 0;
    const int direct_from = HAS_DN ? sm.tab[3 * E + 1] : INT_MAX;
    uint32_t nk = 0;  // TMA thread: k-blocks whose loads this CTA issued (rank 0: armed and issued)
    auto is_dn = [&](int t) { return MODE == 2 || (MODE == 3 && t >= N_up); };
    auto decode = [&](int t) {
        return is_dn(t) ? decode_pair_down(t - N_up, sm.tab, E, nN_dn, p.items_down, rank, s.down_n_outer_items)
                        : decode_pair_up(t, tab_up, E, p.items_up, rank, FUSED ? eid_up : nullptr);
    };

    if (gemm_cta) {
        if (warp == 0 && lane == 0) {
            // ---------------- TMA producer (both CTAs): own A rows + own half of B ----------------
            // Rank 0 arms its full barrier with the stage's bytes of both CTAs; rank 1's loads
            // complete on that barrier (cta_group::2), so the UMMA issuer waits on one barrier per
            // stage.
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            int ready_x = -1;  // fused dispatch: the expert whose rows are known to be copied
            int ready_h = -1;  // fused GEMMs: the expert whose hidden rows are known to be complete
            bool up_done = !HAS_UP, dn_started = false;
            const bool stall = (s.flags & (rank == 0 ? MOE_TEST_STALL_PIPE0 : MOE_TEST_STALL_PIPE1)) != 0;
            // rank 0: the next tile (fused: SwiGLU tiles first, down-projection tiles for producers)
            auto claim = [&]() -> int {
                if (!FUSED) return atomicAdd(&p.meta[(MODE == 1) ? META_TILES_UP : META_TILES_DOWN], 1);
                if (!up_done) {
                    const int v = atomicAdd(&p.meta[META_TILES_UP], 1);
                    if (v < N_up) return v;
                    up_done = true;
                }
                if (producer) {
                    const int v = atomicAdd(&p.meta[META_TILES_DOWN], 1);
                    if (v < N_dn) return N_up + v;
                }
                return total;
            };
            int t = (rank == 0 && !bad) ? claim() : 0;
            for (int j = 0; ok && !bad; ++j) {
                const int slot = j % PAIR_TILE_Q;
                if (rank == 0) {
                    if (!mbar_wait(&sm.tq_empty[slot], ((uint32_t)(j / PAIR_TILE_Q) & 1u) ^ 1u, tmo, sm.abort)) {
                        ok = false;
                        break;
                    }
                    const int v = t < total ? t : -1;
                    sm.tq[slot] = v;
                    mbar_arrive(&sm.tq_full[slot]);
                    st_async_u32(mapa_shared(smem_u32(const_cast<int*>(sm.tq + slot)), 1u), (uint32_t)v,
                                 mapa_shared(smem_u32(&sm.tq_full[slot]), 1u));
                } else {
                    t = pair_tile_wait(sm, j, tmo);
                    if (t == TILE_ABORT) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&sm.tq_full[slot], 4);  // armed for the slot's next use
                }
                if (t < 0 || t >= total) break;
                const bool dn = is_dn(t);
                const TileRef tr = decode(t);
                if (HAS_UP && dispatch && !dn && tr.e != ready_x) {
                    if (!wait_expert_rows(s, p, tr.e, sm.abort, 30 + (int)rank)) {
                        ok = false;
                        break;
                    }
                    ready_x = tr.e;
                }
                if (FUSED && dn && tr.e != ready_h) {
                    // the expert's hidden rows are complete once every SwiGLU tile quarter of the
                    // expert has published (stores completed, async proxy fenced, release add)
                    const uint32_t need = (uint32_t)xexp[tr.e];
                    const unsigned long long t0 = globaltimer();
                    while (ld_acquire_gpu(p.xready + tr.e) < need) {
                        if (*sm.abort || globaltimer() - t0 > tmo) {
                            if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 20 + (int)rank);
                            ok = false;
                            break;
                        }
                        __nanosleep(128);
                    }
                    if (!ok) break;
                    fence_proxy_async_global();  // the TMA loads below read what the acquire ordered
                    ready_h = tr.e;
                    if (rank == 0 && !dn_started) {
                        dn_started = true;
                        atomicMin(&p.trace[MOE_TRACE_GEMM2_START], globaltimer());
                    }
                }
                const int brow = dn ? tr.n * 2 * BN1 + (int)rank * BN1 : tr.n * BN1;
                const CUtensorMap* ta = (FUSED && dn) ? mA2 : mA;
                const CUtensorMap* tb = (FUSED && dn) ? mB2 : (rank == 0 ? mB0 : mB1);
                const int KB = dn ? KB_dn : KB_up;
                const int claim_kb = KB > 8 ? KB - 8 : 0;
                const uint32_t bytes = 2 * (PAIR_A_BYTES + PAIR_B_BYTES);
                int next = total;
                for (int kb = 0; kb < KB; ++kb) {
                    if (stall && j == 0 && kb == KB / 2) {
                        // test hook: this CTA stops issuing, as a stuck load stream would; the
                        // pair's bounded waits run out and the abort path settles what is in flight
                        const unsigned long long t0 = globaltimer();
                        while (!*sm.abort && globaltimer() - t0 < tmo) __nanosleep(1000);
                        ok = false;
                        break;
                    }
                    if (rank == 0 && kb == claim_kb) next = claim();
                    if (!mbar_wait(&sm.empty[st], ph ^ 1u, tmo, sm.abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t* a = sm.stages + st * PAIR_STAGE_BYTES;
                    uint8_t* b = a + PAIR_A_BYTES;
                    if (rank == 0) {
                        mbar_arrive_expect_tx(&sm.full[st], bytes);
                        tma_load_2d(a, ta, &sm.full[st], kb * BK, tr.row >= 0 ? tr.row : s.PC_max);  // 128 compact rows
                        tma_load_3d(b, tb, &sm.full[st], kb * BK, brow, tr.e);  // gate rows / W2 rows 0-127
                    } else {
                        const uint32_t full0 = mapa_shared(smem_u32(&sm.full[st]), 0u);
                        // an odd CTA without rows loads a box past the last row: zeros, so its idle
                        // half of the UMMA multiplies zeros (less switching power than stale rows)
                        tma_load_2d_pair(a, ta, full0, kb * BK, tr.row >= 0 ? tr.row : s.PC_max);
                        tma_load_3d_pair(b, tb, full0, kb * BK, brow, tr.e);  // up rows / W2 rows 128-255
                    }
                    ++nk;
                    if (++st == PAIR_STAGES) {
                        st = 0;
                        ph ^= 1u;
                    }
                }
                if (rank == 0) t = next;
            }
            if (!ok) {  // the loads still in flight are settled below, once both CTAs have stopped
                if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 10 + (int)rank);
                pair_abort(sm, rank);
            }
        } else if (warp == 1 && lane == 0) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            if (rank == 0) {
                // ---------------- UMMA issuer (rank 0) ----------------
                if (bad) {
                    set_status(p.meta, ST_PAIR_TMEM, (int)*sm.peer_base);
                    pair_abort(sm, rank);
                }
                const uint32_t idesc = umma_idesc_bf16(2 * BM, 2 * BN1);
                int b = 0;
                uint32_t aph = 0;
                for (int j = 0; ok && !bad; ++j) {
                    const int t = pair_tile_wait(sm, j, tmo);
                    if (t == TILE_ABORT) {
                        ok = false;
                        break;
                    }
                    mbar_arrive(&sm.tq_empty[j % PAIR_TILE_Q]);
                    if (t < 0) break;
                    const int KB = is_dn(t) ? KB_dn : KB_up;
                    if (!mbar_wait_cluster(&sm.acc_empty[b], aph ^ 1u, tmo, sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dt = tmem + (uint32_t)(b * 256);
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!mbar_wait_cluster(&sm.full[st], ph, tmo, sm.abort)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(sm.stages + st * PAIR_STAGE_BYTES);
                        const uint64_t ad = sdesc_sw128(a_addr);
                        const uint64_t bd = sdesc_sw128(a_addr + PAIR_A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_bf16_pair(dt, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                        umma_commit_pair(&sm.empty[st], 0x3);
                        if (++st == PAIR_STAGES) {
                            st = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit_pair(&sm.acc_full[b], 0x3);
                    b ^= 1;
                    if (b == 0) aph ^= 1u;
                }
                // Final commit to both CTAs' drain barrier: every UMMA issued has completed when it
                // fires.
                umma_commit_pair(sm.drain, 0x3);
            }
            if (!ok) {
                if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 12 + (int)rank);
                pair_abort(sm, rank);
            }
            int never = 0;
            if (!mbar_wait(sm.drain, 0, tmo, &never) && !*sm.abort)
                set_status(p.meta, ST_PIPE_TIMEOUT, 14 + (int)rank);
        } else if (warp >= 2) {
            // ---------------- epilogue (both CTAs): this CTA's 128 rows ----------------
            const int q = warp & 3;
            const bool flags = HAS_DN && overlapped;
            if (HAS_UP && dispatch) dispatch_rows(s, p);
            EpiStage es{sm.epi + (warp - 2) * 2 * EPI_CHUNK_BYTES, 0};
            const uint32_t acc_empty0 = mapa_shared(smem_u32(sm.acc_empty), 0u);
            int b = 0;
            uint32_t aph = 0;
            for (int j = 0; !bad; ++j) {
                int t = 0;
                if (lane == 0) {
                    t = pair_tile_wait(sm, j, tmo);
                    if (t != TILE_ABORT && rank == 0) mbar_arrive(&sm.tq_empty[j % PAIR_TILE_Q]);
                }
                t = __shfl_sync(0xffffffffu, t, 0);
                if (t == TILE_ABORT) {
                    if (lane == 0) {
                        if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 18 + (int)rank);
                        pair_abort(sm, rank);
                    }
                    break;
                }
                if (t < 0) break;
                const bool dn = is_dn(t);
                const TileRef tr = decode(t);
                if (!mbar_wait(&sm.acc_full[b], aph, tmo, sm.abort)) {
                    if (!*sm.abort) set_status(p.meta, ST_PIPE_TIMEOUT, 16 + (int)rank);
                    if (lane == 0) pair_abort(sm, rank);
                    break;
                }
                tc_fence_after();
                const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * 256);
                const int c0 = tr.row + q * 32;  // this warp's first compact row (tr.row < 0: no rows)
                DownRow dr{nullptr, -1, -1, false};
                if (dn) {
                    if (tr.row >= 0) dr = down_row(s, p, c0 + lane, MT, direct_from);
                    epilogue_down(es, FUSED ? mOut2 : mOut, tb, tr.n, 2 * BN1, dr, lane);
                } else {
                    epilogue_swiglu(es, mOut, tb, tr.n, c0, tr.row >= 0, lane);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(acc_empty0 + b * 8u);
                if (dn) {
                    if (flags) publish_rows(s, p, dr, tr.n, lane);
                    const bool stored = __any_sync(0xffffffffu, dr.band >= 0);
                    if (lane == 0 && stored) last_end = globaltimer();
                }
                if (FUSED && !dn && lane == 0) {
                    // this warp's quarter of the SwiGLU tile (stored or idle) counts towards its
                    // expert's hidden rows being complete: stores complete, async proxy fenced, release
                    bulk_wait_all();
                    fence_proxy_async_global();
                    __threadfence();
                    red_release_gpu_add(p.xready + tr.e, 1u);
                }
                b ^= 1;
                if (b == 0) aph ^= 1u;
            }
            if (lane == 0) bulk_wait_all();  // staging buffers stay valid until every store is done
            __syncwarp();
        }
        __syncwarp();
        tc_fence_before();
        cluster_sync();  // both CTAs: all roles done, all UMMAs complete (drain), no remote access left
        // Every abort word write (pair_abort sets both CTAs') came before that barrier, so both CTAs
        // take this branch or neither. Rank 1 hands its count of issued k-blocks to rank 0, which
        // settles every load still in flight before either CTA goes on.
        if (*sm.abort) {
            if (warp == 0 && lane == 0 && rank == 1)
                st_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(sm.peer_k)), 0u), nk);
            cluster_sync();
            if (warp == 0 && lane == 0 && rank == 0) pair_settle(sm, nk, *sm.peer_k, tmo);
            cluster_sync();
        }
        if (warp == 1) {
            __syncwarp();
            tc_fence_after();
            tmem_dealloc_pair(tmem, TMEM_COLS);
        }
        __syncwarp();
        cluster_sync();  // neither CTA goes on (or leaves) while the pair's TMEM release is in progress
        if (HAS_DN && warp >= 2 && lane == 0 && last_end) atomicMax(&p.trace[MOE_TRACE_GEMM2_END], last_end);
        clock_span_add(p, clk, MODE == 2 ? MOE_TRACE_DOWN_CYCLES : MOE_TRACE_UP_CYCLES);
    }
    // copy engines: consumer CTAs from the start (fused: after their SwiGLU tiles), producers once
    // their tiles are done (tail assist)
    if (HAS_DN && overlapped && (!producer || (s.flags & MOE_TAIL_ASSIST)))
        copy_units(s, p, sm.stages, sm.cbar, sm.abort, META_QUEUE, true, stall, direct_from);
}

template <int MODE>  // 1: SwiGLU up-projection -> Hc; 2: down-projection -> Yp (+ flags / consumers)
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    gemm_pair_kernel(Shape s, PlanPtrs p, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                     const __grid_constant__ CUtensorMap tmOut, int num_producers, int overlapped) {
    pair_body<MODE>(s, p, &tmA, &tmB0, &tmB1, &tmOut, nullptr, nullptr, nullptr, num_producers, overlapped);
}

// Both expert GEMMs in one launch (MOE_FUSED_GEMMS): the MODE 3 body.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    gemm_fused_pair_kernel(Shape s, PlanPtrs p, const __grid_constant__ CUtensorMap tmXc,
                           const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW3,
                           const __grid_constant__ CUtensorMap tmHcOut, const __grid_constant__ CUtensorMap tmHc,
                           const __grid_constant__ CUtensorMap tmW2h, const __grid_constant__ CUtensorMap tmYpOut,
                           int num_producers) {
    pair_body<3>(s, p, &tmXc, &tmW1, &tmW3, &tmHcOut, &tmHc, &tmW2h, &tmYpOut, num_producers, 1);
}

static cudaError_t set_smem_attr(const void* fn) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM);
}

cudaError_t launch_gemm_swiglu(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmW1,
                               const CUtensorMap& tmW3, const CUtensorMap& tmOut, int sms, cudaStream_t st) {
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(&gemm_kernel<1>));
    if (e != cudaSuccess) return e;
    return launch_k(gemm_kernel<1>, dim3(sms), dim3(GEMM_THREADS), GEMM_SMEM, st, (s.flags & MOE_PDL) != 0, s, p, tmA,
                    tmW1, tmW3, tmOut, sms, 0);
}

// Co-resident clusters of two of a pair kernel on this device (cluster occupancy query, cached).
template <int MODE>
static cudaError_t pair_clusters(int* out) {
    const void* fn = reinterpret_cast<const void*>(&gemm_pair_kernel<MODE>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, PAIR_SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int cache[64] = {0};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (cache[dev] == 0) {
        cudaLaunchConfig_t q = {};  // the cluster size (2) is the kernel's compile-time one
        q.gridDim = dim3(2, 1, 1);
        q.blockDim = dim3(GEMM_THREADS, 1, 1);
        q.dynamicSmemBytes = PAIR_SMEM;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &q);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        cache[dev] = n;
    }
    *out = cache[dev];
    return cudaSuccess;
}

cudaError_t launch_gemm_swiglu_pair(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA,
                                    const CUtensorMap& tmW1, const CUtensorMap& tmW3, const CUtensorMap& tmOut,
                                    cudaStream_t st) {
    int pairs = 0;
    cudaError_t e = pair_clusters<1>(&pairs);
    if (e != cudaSuccess) return e;
    return launch_k(gemm_pair_kernel<1>, dim3(2 * pairs), dim3(GEMM_THREADS), PAIR_SMEM, st, (s.flags & MOE_PDL) != 0,
                    s, p, tmA, tmW1, tmW3, tmOut, 2 * pairs, 0);
}

// Down-projection on CTA pairs: 2 x (co-resident clusters) CTAs, the last `consumers` (even) of them
// consumer CTAs when overlapped. Every tile is handed out by the counter, so no CTA waits for a
// particular one to become resident: no cooperative launch is needed.
cudaError_t launch_gemm_down_pair(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmW2h,
                                  const CUtensorMap& tmOut, int consumers, bool overlapped, cudaStream_t st) {
    int pairs = 0;
    cudaError_t e = pair_clusters<2>(&pairs);
    if (e != cudaSuccess) return e;
    const int grid = 2 * pairs, producers = overlapped ? grid - consumers : grid;
    if ((consumers & 1) || producers < 2) return cudaErrorInvalidConfiguration;
    return launch_k(gemm_pair_kernel<2>, dim3(grid), dim3(GEMM_THREADS), PAIR_SMEM, st, (s.flags & MOE_PDL) != 0, s, p,
                    tmA, tmW2h, tmW2h, tmOut, producers, overlapped ? 1 : 0);
}

cudaError_t launch_gemm_fused_pair(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmXc, const CUtensorMap& tmW1,
                                   const CUtensorMap& tmW3, const CUtensorMap& tmHcOut, const CUtensorMap& tmHc,
                                   const CUtensorMap& tmW2h, const CUtensorMap& tmYpOut, int consumers,
                                   cudaStream_t st) {
    const void* fn = reinterpret_cast<const void*>(&gemm_fused_pair_kernel);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, PAIR_SMEM_FUSED);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int cache[64] = {0};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (cache[dev] == 0) {
        cudaLaunchConfig_t q = {};  // the cluster size (2) is the kernel's compile-time one
        q.gridDim = dim3(2, 1, 1);
        q.blockDim = dim3(GEMM_THREADS, 1, 1);
        q.dynamicSmemBytes = PAIR_SMEM_FUSED;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &q);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        cache[dev] = n;
    }
    const int grid = 2 * cache[dev], producers = grid - consumers;
    if ((consumers & 1) || producers < 2) return cudaErrorInvalidConfiguration;
    return launch_k(gemm_fused_pair_kernel, dim3(grid), dim3(GEMM_THREADS), PAIR_SMEM_FUSED, st,
                    (s.flags & MOE_PDL) != 0, s, p, tmXc, tmW1, tmW3, tmHcOut, tmHc, tmW2h, tmYpOut, producers);
}

cudaError_t launch_gemm_down(const Shape& s, const PlanPtrs& p, const CUtensorMap& tmA, const CUtensorMap& tmW2,
                             const CUtensorMap& tmOut, int sms, int consumers, bool overlapped, cudaStream_t st) {
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(&gemm_kernel<2>));
    if (e != cudaSuccess) return e;
    const int producers = overlapped ? sms - consumers : sms;
    int ov = overlapped ? 1 : 0;
    const int threads = (overlapped && (s.flags & MOE_COPY_WARPS)) ? GEMM_THREADS_MAX : GEMM_THREADS;
    Shape sa = s;
    PlanPtrs pa = p;
    CUtensorMap a = tmA, b0 = tmW2, b1 = tmW2, o = tmOut;
    if (!overlapped) {
        gemm_kernel<2><<<sms, GEMM_THREADS, GEMM_SMEM, st>>>(sa, pa, a, b0, b1, o, producers, ov);
        return cudaGetLastError();
    }
    // Cooperative launch: every CTA (producers and consumers) is resident at once, or the launch
    // fails; the consumers' waits on producer flags can therefore always be satisfied.
    void* args[] = {&sa, &pa, &a, &b0, &b1, &o, (void*)&producers, &ov};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&gemm_kernel<2>), dim3(sms), dim3(threads),
                                       args, GEMM_SMEM, st);
}

// Sequential return copy: every SM takes copy units, no flags ([TLS Figure 9 caption] baseline).
__global__ void __launch_bounds__(GEMM_THREADS, 1) copy_seq_kernel(Shape s, PlanPtrs p) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm = carve_smem(smem_raw);
    if (threadIdx.x == 0) {
        for (int i = 0; i < COPY_NBUF; ++i) mbar_init(&sm.cbar[i], 1);
        *sm.abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    copy_units(s, p, sm.stages, sm.cbar, sm.abort, META_QUEUE_SEQ, false, 0u, INT_MAX);
}

cudaError_t launch_copy_seq(const Shape& s, const PlanPtrs& p, int sms, cudaStream_t st) {
    cudaError_t e = set_smem_attr(reinterpret_cast<const void*>(&copy_seq_kernel));
    if (e != cudaSuccess) return e;
    copy_seq_kernel<<<sms, GEMM_THREADS, GEMM_SMEM, st>>>(s, p);
    return cudaGetLastError();
}

}  // namespace moe
