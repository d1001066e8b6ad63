// Row-band copy engine of the return path: Yp rows -> the owner's slice of Ret.
//
// "Fine-grained Computation-Communication Overlap via Tile-level Signaling and Scheduling for
// Mixture-of-Experts" (pith.science/paper/W2ZARMHG), "Core claim": the consumer polls the tile
// flags and issues one contiguous write per row-band segment. On one GPU the write is an
// HBM-to-HBM copy. Every warp of a copying CTA is an independent copy engine: it takes a work unit,
// waits for the unit's flags, and moves the rows through two shared-memory buffers with TMA bulk
// copies (global -> shared completes on an mbarrier, shared -> global is a bulk group), so each
// warp keeps two loads in flight and a 6-warp CTA about 192 KB.
//
// Work units: band (schedule position) x row chunk of rows_per_unit rows, handed out in schedule
// order by an atomic counter, so idle engines always take the oldest outstanding band.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Per-warp copy engine: two COPY_PIECE staging buffers and their mbarriers. Lane 0 issues.
struct CopyEngine {
    uint8_t* buf;         // 2 * COPY_PIECE bytes, 1024-byte aligned
    uint64_t* bar;        // 2 mbarriers, count 1
    uint32_t phase_bits;  // parity to wait for next, per buffer
    uint32_t pending;     // buffers with a load in flight that has not been waited for
};

// Lane 0 only. Copies `bytes` (a multiple of 16) from src to dst, keeping two bulk loads in
// flight. Returns false on timeout.
__device__ __forceinline__ bool engine_copy(CopyEngine& ce, const uint8_t* src, uint8_t* dst, size_t bytes,
                                            unsigned long long timeout_ns, volatile int* abort) {
    const int np = (int)((bytes + COPY_PIECE - 1) / COPY_PIECE);
    bulk_wait_read_all();  // every earlier store of this lane has finished reading its buffer
    auto piece = [&](int i) { return (uint32_t)min((size_t)COPY_PIECE, bytes - (size_t)i * COPY_PIECE); };
    auto issue = [&](int i) {
        const int b = i & 1;
        mbar_arrive_expect_tx(&ce.bar[b], piece(i));
        bulk_load(ce.buf + (size_t)b * COPY_PIECE, src + (size_t)i * COPY_PIECE, piece(i), &ce.bar[b]);
        ce.pending |= 1u << b;
    };
    for (int i = 0; i < min(np, 2); ++i) issue(i);
    for (int i = 0; i < np; ++i) {
        const int b = i & 1;
        if (!mbar_wait(&ce.bar[b], (ce.phase_bits >> b) & 1u, timeout_ns, abort)) return false;
        ce.phase_bits ^= 1u << b;
        ce.pending &= ~(1u << b);
        bulk_store(dst + (size_t)i * COPY_PIECE, ce.buf + (size_t)b * COPY_PIECE, piece(i));
        bulk_commit();
        if (i + 2 < np) {
            bulk_wait_read_all();  // store i has read buffer b
            issue(i + 2);
        }
    }
    return true;
}

// Lane 0, before the CTA leaves: wait (bounded) for loads still in flight, then for all stores.
__device__ __forceinline__ void engine_drain(CopyEngine& ce, unsigned long long timeout_ns) {
    int never = 0;
    for (int b = 0; b < 2; ++b)
        if (ce.pending & (1u << b)) {
            mbar_wait(&ce.bar[b], (ce.phase_bits >> b) & 1u, timeout_ns, &never);
            ce.phase_bits ^= 1u << b;
        }
    ce.pending = 0;
    bulk_wait_all();
}

// Called by every thread of the CTA. Each warp is an independent copy engine with its own slice of
// the staging area (`ring`, COPY_WARPS * 2 * COPY_PIECE bytes) and two of the mbarriers in `bars`;
// it takes units from meta[queue] until none is left. wait_flags: acquire every tile flag of the
// unit's segment (== want) before copying.
__device__ void copy_units(const Shape& s, const PlanPtrs& p, uint8_t* ring, uint64_t* bars, volatile int* s_abort,
                           int queue, bool wait_flags, uint32_t want) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int MT = p.meta[META_MTILES];
    if (MT < 0 || MT > s.MT_max) MT = 0;
    const int units = MT * s.units_per_band;
    const size_t rowb = (size_t)s.d * 2;
    CopyEngine ce{ring + (size_t)warp * 2 * COPY_PIECE, bars + 2 * warp, 0u, 0u};
    unsigned long long t_first = ~0ull;
    bool did = false;

    for (;;) {
        int u = 0;
        if (lane == 0) u = atomicAdd(&p.meta[queue], 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        if (__any_sync(0xffffffffu, *s_abort != 0) || u >= units) break;
        const int pos = u / s.units_per_band, c = u - pos * s.units_per_band;
        const int m = p.sched[pos];
        const int row0 = p.tiles[4 * m + 2], valid = p.tiles[4 * m + 3];
        const int rb = c * s.rows_per_unit;
        if (rb >= valid) continue;
        const int re = min(valid, rb + s.rows_per_unit);

        if (wait_flags) {
            const int first = p.seg[2 * pos], nb = p.seg[2 * pos + 1];
            const int nf = nb * s.n_tiles_n2;
            bool failed = false;
            for (int f = lane; f < nf && !failed; f += 32) {
                const int mb = p.sched[first + f / s.n_tiles_n2];
                const uint32_t* fl = p.flags + (size_t)mb * s.n_tiles_n2 + (f % s.n_tiles_n2);
                if (ld_acquire_gpu(fl) == want) continue;
                const unsigned long long t0 = globaltimer();
                for (;;) {
                    __nanosleep(32);
                    if (ld_acquire_gpu(fl) == want) break;
                    if (*s_abort) {
                        failed = true;
                        break;
                    }
                    if (globaltimer() - t0 > s.timeout_ns) {
                        *s_abort = 1;
                        set_status(p.meta, ST_FLAG_TIMEOUT, mb);
                        failed = true;
                        break;
                    }
                }
            }
            if (__any_sync(0xffffffffu, failed)) break;
        }
        if (lane == 0) {
            if (!did) t_first = globaltimer();
            did = true;
            fence_proxy_async_global();
            const uint8_t* src = reinterpret_cast<const uint8_t*>(p.Yp) + (size_t)(row0 + rb) * rowb;
            uint8_t* dst = reinterpret_cast<uint8_t*>(p.Ret) + (size_t)(p.tile_ret[m] + rb) * rowb;
            if (!engine_copy(ce, src, dst, (size_t)(re - rb) * rowb, s.timeout_ns, s_abort)) {
                *s_abort = 1;
                set_status(p.meta, ST_COPY_TIMEOUT, m);
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        engine_drain(ce, s.timeout_ns);
        if (did) {
            atomicMin(&p.trace[MOE_TRACE_COPY_START], t_first);
            atomicMax(&p.trace[MOE_TRACE_COPY_END], globaltimer());
        }
    }
    __syncwarp();
}

}  // namespace moe
