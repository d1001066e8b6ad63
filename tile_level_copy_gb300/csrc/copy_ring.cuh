// Row-band copy engines of the return path: Yp rows -> the owner's slice of Ret.
//
// "Fine-grained Computation-Communication Overlap via Tile-level Signaling and Scheduling for
// Mixture-of-Experts" (pith.science/paper/W2ZARMHG), "Core claim": the consumer polls the tile
// flags and issues one contiguous write per row-band segment. On one GPU the write is an
// HBM-to-HBM copy, and the poll reads one counter per band, to which every epilogue warp that stored
// rows of the band release-adds their number beside its tile flag (ready at valid rows x tiles per
// band).
//
// Bulk engine (copy_units): every warp of a copying CTA takes a work unit, waits for the unit's
// bands, and moves the rows through two shared-memory buffers with TMA bulk copies (global ->
// shared completes on an mbarrier, shared -> global is a bulk group), keeping two 16 KB loads in
// flight, also across unit boundaries. SIMT engine (copy_units_simt): one warp moving rows through
// registers with 16-byte loads and stores, no shared memory, for the extra warps of producer CTAs.
//
// Work units: band (hand-out position) x row chunk of rows_per_unit rows, handed out in the
// down-projection's hand-out order by an atomic counter, so idle engines always take the oldest
// outstanding band.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Per-warp copy engine: two COPY_PIECE staging buffers used in FIFO order, their mbarriers, and
// the destination of the piece each holds. Lane 0 issues all bulk operations; pieces flow through
// the two buffers continuously, across unit boundaries.
struct CopyEngine {
    uint8_t* buf;         // 2 * COPY_PIECE bytes, 1024-byte aligned
    uint64_t* bar;        // 2 mbarriers, count 1
    uint8_t* dst[2];      // destination of the piece loaded into each buffer
    uint32_t len[2];
    uint32_t phase_bits;  // parity to wait for next, per buffer
    int head, count;      // oldest occupied buffer, occupied buffers
};

// Lane 0: wait for the oldest load, store it out. Returns false on timeout.
__device__ __forceinline__ bool engine_retire(CopyEngine& ce, unsigned long long timeout_ns, volatile int* abort) {
    const int b = ce.head;
    if (!mbar_wait(&ce.bar[b], (ce.phase_bits >> b) & 1u, timeout_ns, abort)) return false;
    ce.phase_bits ^= 1u << b;
    bulk_store(ce.dst[b], ce.buf + (size_t)b * COPY_PIECE, ce.len[b]);
    bulk_commit();
    ce.head ^= 1;
    --ce.count;
    return true;
}

// Lane 0: queue one piece (len <= COPY_PIECE, a multiple of 16). Returns false on timeout.
__device__ __forceinline__ bool engine_push(CopyEngine& ce, const uint8_t* src, uint8_t* dst, uint32_t len,
                                            unsigned long long timeout_ns, volatile int* abort) {
    if (ce.count == 2 && !engine_retire(ce, timeout_ns, abort)) return false;
    const int b = ce.head ^ ce.count;  // next free buffer in FIFO order
    bulk_wait_read_all();              // the store that last used buffer b has read it
    ce.dst[b] = dst;
    ce.len[b] = len;
    mbar_arrive_expect_tx(&ce.bar[b], len);
    bulk_load(ce.buf + (size_t)b * COPY_PIECE, src, len, &ce.bar[b]);
    ++ce.count;
    return true;
}

// Lane 0: store every piece that is loaded (before the engine waits on a band that is not ready,
// so finished data does not sit in shared memory meanwhile). Returns false on timeout.
__device__ __forceinline__ bool engine_flush(CopyEngine& ce, unsigned long long timeout_ns, volatile int* abort) {
    while (ce.count > 0)
        if (!engine_retire(ce, timeout_ns, abort)) return false;
    return true;
}

// Lane 0, before the CTA leaves: store what is still loaded, then wait for every store. The
// waits are bounded; after a timeout the remaining loads are still waited for (bounded) so that
// no copy into shared memory is in flight when the CTA exits.
__device__ __forceinline__ void engine_drain(CopyEngine& ce, unsigned long long timeout_ns) {
    int never = 0;
    while (ce.count > 0)
        if (!engine_retire(ce, timeout_ns, &never)) {
            ce.head ^= 1;
            --ce.count;
        }
    bulk_wait_all();
}

// Bounds check of the plan entries one copy unit reads (hand-out position pos -> band m, its rows
// in Yp and Ret, and the bands of its segment with their valid rows). A failure is reported as
// ST_BAD_PLAN and the copy stops, so a corrupt plan never turns into an out-of-range access.
__device__ __forceinline__ bool copy_unit_ok(const Shape& s, const PlanPtrs& p, int MT, int pos, bool wait_flags) {
    const int m = p.order[pos];
    if (m < 0 || m >= MT) return false;
    const int row0 = p.tiles[4 * m + 2], valid = p.tiles[4 * m + 3], ret0 = p.tile_ret[m];
    if (valid < 1 || valid > s.tbM || row0 < 0 || row0 + valid > s.P_max || ret0 < 0 || ret0 + valid > s.T * s.k)
        return false;
    if (wait_flags) {
        const int first = p.seg[2 * pos], nb = p.seg[2 * pos + 1];
        if (first < 0 || nb < 1 || nb > s.mgb || first + nb > MT) return false;
        for (int i = 0; i < nb; ++i) {
            const int b = p.order[first + i];
            if (b < 0 || b >= MT || p.tiles[4 * b + 3] < 1 || p.tiles[4 * b + 3] > s.tbM) return false;
        }
    }
    return true;
}

// Count at which band b's counter says that every row of every N tile of the band is stored
// (stall = 1: a count it never reaches, the stalled-consumer test hook).
__device__ __forceinline__ uint32_t band_ready(const Shape& s, const PlanPtrs& p, int b, uint32_t stall) {
    return (uint32_t)p.tiles[4 * b + 3] * (uint32_t)s.n_tiles_n2 + stall;
}

// Called by every thread of the CTA. Each warp is an independent copy engine with its own slice of
// the staging area (`ring`, COPY_WARPS * 2 * COPY_PIECE bytes) and two of the mbarriers in `bars`;
// it takes units from meta[queue] until none is left. wait_flags: acquire the band counter of every
// band of the unit's segment (== band_ready: all rows of all tiles of the band published) before
// copying. An engine claims its next unit only once the current one is acquired (never while it
// waits on a band), and the next unit's counters are polled while the previous unit's pieces are
// still in flight.
// skip_item: bands whose last row's down-projection work item is at or past this index are returned
// by the GEMM's own epilogue (MOE_DIRECT_TAIL): their counters are not waited for, and an engine that
// reaches one of their units stops (they are the last hand-out positions).
__device__ void copy_units(const Shape& s, const PlanPtrs& p, uint8_t* ring, uint64_t* bars, volatile int* s_abort,
                           int queue, bool wait_flags, uint32_t stall, int skip_item) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int MT = p.meta[META_MTILES];
    if (MT < 0 || MT > s.MT_max) MT = 0;
    const int units = copy_unit_count(s, MT);
    const size_t rowb = (size_t)s.d * 2;
    CopyEngine ce{};
    ce.buf = ring + (size_t)warp * 2 * COPY_PIECE;
    ce.bar = bars + 2 * warp;
    unsigned long long t_first = ~0ull, t_acq = 0, t_load = 0;
    bool did = false;

    int u_next = 0;
    if (lane == 0) u_next = atomicAdd(&p.meta[queue], 1);
    for (;;) {
        const int u = __shfl_sync(0xffffffffu, u_next, 0);
        if (__any_sync(0xffffffffu, *s_abort != 0) || u >= units) break;
        int pos, rb, rpu;
        copy_unit_decode(s, MT, u, &pos, &rb, &rpu);
        if (!__all_sync(0xffffffffu, copy_unit_ok(s, p, MT, pos, wait_flags))) {
            if (lane == 0) {
                set_status(p.meta, ST_BAD_PLAN, pos);
                *s_abort = 1;
            }
            break;
        }
        const int m = p.order[pos];
        const int row0 = p.tiles[4 * m + 2], valid = p.tiles[4 * m + 3];
        // the bands the epilogue returns are a suffix of the hand-out positions (band_item does not
        // decrease along them), so every unit from here on is theirs: stop instead of claiming them
        if (p.band_item[m] >= skip_item) break;
        if (rb >= valid) {
            if (lane == 0) u_next = atomicAdd(&p.meta[queue], 1);
            continue;
        }
        const int re = min(valid, rb + rpu);

        if (wait_flags) {
            // lane 0 acquires the counter of every band of the unit's segment (all its tiles done)
            bool failed = false;
            if (lane == 0) {
                const int first = p.seg[2 * pos], nb = p.seg[2 * pos + 1];
                for (int i = 0; i < nb && !failed; ++i) {
                    const int b = p.order[first + i];
                    if (p.band_item[b] >= skip_item) continue;  // returned by the epilogue
                    const uint32_t* bc = p.bands + b;
                    const uint32_t want = band_ready(s, p, b, stall);
                    if (ld_acquire_gpu(bc) == want) continue;
                    if (!engine_flush(ce, s.timeout_ns, s_abort)) {
                        *s_abort = 1;
                        set_status(p.meta, ST_COPY_TIMEOUT, m);
                        failed = true;
                        break;
                    }
                    const unsigned long long t0 = globaltimer();
                    for (;;) {
                        __nanosleep(100);
                        if (ld_acquire_gpu(bc) == want) break;
                        if (*s_abort) {
                            failed = true;
                            break;
                        }
                        if (globaltimer() - t0 > s.timeout_ns) {
                            *s_abort = 1;
                            set_status(p.meta, ST_FLAG_TIMEOUT, p.order[first + i]);
                            failed = true;
                            break;
                        }
                    }
                }
            }
            if (__any_sync(0xffffffffu, failed)) break;
            if (lane == 0) t_acq = globaltimer();
        }
        // The next unit is claimed only now that this one is ready, so a unit queued behind a band
        // that is still being computed is never held by an engine waiting on that band; the claim
        // is in flight while this unit's rows move.
        if (lane == 0) u_next = atomicAdd(&p.meta[queue], 1);
        if (lane == 0) {
            if (!did) t_first = globaltimer();
            did = true;
            fence_proxy_async_global();
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.Yp) + (size_t)(row0 + rb) * rowb;
            uint8_t* dst = reinterpret_cast<uint8_t*>(p.Ret) + (size_t)(p.tile_ret[m] + rb) * rowb;
            const size_t bytes = (size_t)(re - rb) * rowb;
            for (size_t o = 0; o < bytes; o += COPY_PIECE) {
                const uint32_t len = (uint32_t)min((size_t)COPY_PIECE, bytes - o);
                if (!engine_push(ce, src + o, dst + o, len, s.timeout_ns, s_abort)) {
                    *s_abort = 1;
                    set_status(p.meta, ST_COPY_TIMEOUT, m);
                    break;
                }
            }
            t_load = globaltimer();
        }
        __syncwarp();
    }
    if (lane == 0) {
        const unsigned long long t_drain = globaltimer();
        engine_drain(ce, s.timeout_ns);
        if (did) {
            atomicMin(&p.trace[MOE_TRACE_COPY_START], t_first);
            atomicMax(&p.trace[MOE_TRACE_COPY_END], globaltimer());
            atomicMax(&p.trace[MOE_TRACE_LAST_LOAD], t_load);
            atomicMax(&p.trace[MOE_TRACE_LAST_DRAIN], t_drain);
            if (t_acq) atomicMax(&p.trace[MOE_TRACE_LAST_ACQUIRE], t_acq);
        }
    }
    __syncwarp();
}

// SIMT copy engine: one warp, 16-byte loads and stores through registers (16 per lane in flight),
// no shared memory, so it can run beside a producer's GEMM warps in the same CTA. Same queue, same
// band-counter acquire as copy_units; the generic-proxy loads need no proxy fence because producers
// fence their TMA stores into the generic proxy before they release the counter.
__device__ __forceinline__ uint4 ld_cg_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ void st_cg_v4(uint4* p, const uint4& v) {
    asm volatile("st.global.cg.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ void copy_units_simt(const Shape& s, const PlanPtrs& p, volatile int* s_abort, int queue, uint32_t stall,
                                int skip_item) {
    const int lane = threadIdx.x & 31;
    int MT = p.meta[META_MTILES];
    if (MT < 0 || MT > s.MT_max) MT = 0;
    const int units = copy_unit_count(s, MT);
    const size_t rowb = (size_t)s.d * 2;
    unsigned long long t_first = ~0ull, t_acq = 0;
    bool did = false;
    constexpr int UNROLL = 16;

    int u_next = 0;
    if (lane == 0) u_next = atomicAdd(&p.meta[queue], 1);
    for (;;) {
        const int u = __shfl_sync(0xffffffffu, u_next, 0);
        if (__any_sync(0xffffffffu, *s_abort != 0) || u >= units) break;
        int pos, rb, rpu;
        copy_unit_decode(s, MT, u, &pos, &rb, &rpu);
        if (!__all_sync(0xffffffffu, copy_unit_ok(s, p, MT, pos, true))) {
            if (lane == 0) {
                set_status(p.meta, ST_BAD_PLAN, pos);
                *s_abort = 1;
            }
            break;
        }
        const int m = p.order[pos];
        const int row0 = p.tiles[4 * m + 2], valid = p.tiles[4 * m + 3];
        // the bands the epilogue returns are a suffix of the hand-out positions (band_item does not
        // decrease along them), so every unit from here on is theirs: stop instead of claiming them
        if (p.band_item[m] >= skip_item) break;
        if (rb >= valid) {
            if (lane == 0) u_next = atomicAdd(&p.meta[queue], 1);
            continue;
        }
        const int re = min(valid, rb + rpu);
        bool failed = false;
        if (lane == 0) {
            const int first = p.seg[2 * pos], nb = p.seg[2 * pos + 1];
            for (int i = 0; i < nb && !failed; ++i) {
                const int b = p.order[first + i];
                if (p.band_item[b] >= skip_item) continue;  // returned by the epilogue
                const uint32_t* bc = p.bands + b;
                const uint32_t want = band_ready(s, p, b, stall);
                if (ld_acquire_gpu(bc) == want) continue;
                const unsigned long long t0 = globaltimer();
                for (unsigned ns = 64;; ns = ns < 512 ? 2 * ns : ns) {
                    __nanosleep(ns);
                    if (ld_acquire_gpu(bc) == want) break;
                    if (*s_abort) {
                        failed = true;
                        break;
                    }
                    if (globaltimer() - t0 > s.timeout_ns) {
                        *s_abort = 1;
                        set_status(p.meta, ST_FLAG_TIMEOUT, p.order[first + i]);
                        failed = true;
                        break;
                    }
                }
            }
            t_acq = globaltimer();
            if (!did) t_first = t_acq;
            if (!failed) u_next = atomicAdd(&p.meta[queue], 1);  // claimed once this unit is ready
        }
        if (__any_sync(0xffffffffu, failed)) break;
        __syncwarp();  // orders lane 0's acquire before every lane's loads
        did = true;
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(p.Yp) +
                                                          (size_t)(row0 + rb) * rowb);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.Ret) + (size_t)(p.tile_ret[m] + rb) * rowb);
        const int n = (int)((size_t)(re - rb) * rowb / 16);
        for (int base = 0; base < n; base += 32 * UNROLL) {
            uint4 v[UNROLL];
#pragma unroll
            for (int i = 0; i < UNROLL; ++i) {
                const int idx = base + i * 32 + lane;
                if (idx < n) v[i] = ld_cg_v4(src + idx);
            }
#pragma unroll
            for (int i = 0; i < UNROLL; ++i) {
                const int idx = base + i * 32 + lane;
                if (idx < n) st_cg_v4(dst + idx, v[i]);
            }
        }
    }
    __threadfence();  // this lane's stores performed before the completion stamp
    __syncwarp();
    if (lane == 0 && did) {
        const unsigned long long t_end = globaltimer();
        atomicMin(&p.trace[MOE_TRACE_COPY_START], t_first);
        atomicMax(&p.trace[MOE_TRACE_COPY_END], t_end);
        atomicMax(&p.trace[MOE_TRACE_LAST_LOAD], t_end);
        atomicMax(&p.trace[MOE_TRACE_LAST_DRAIN], t_end);
        atomicMax(&p.trace[MOE_TRACE_LAST_ACQUIRE], t_acq);
    }
}

}  // namespace moe
